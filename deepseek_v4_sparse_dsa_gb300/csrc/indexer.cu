// Planning and launch sequence of the DSA indexer score and fused top-k (sm_103a).
//
// The kernel itself is in indexer_kernel.cuh (see there for the design).  This file:
// the host-side plan of a call (tile shapes, pipeline depth, TMEM buffers, workspace
// layout), the one-CTA plan kernel that lays the query groups of a top-k call out on a
// line from the actual context lengths, the tensor maps, and the launch sequence
// plan kernel -> indexer kernel -> merge kernel.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "indexer_kernel.cuh"

namespace dsa {

// Visible key tiles of query group u (its last real query sees the most keys).
__device__ __forceinline__ int group_tiles(const int32_t* context_lens, int u, int ngroups, int nq, int next_n,
                                           int causal, int max_len) {
  const int b = u / ngroups;
  const int gi = u - b * ngroups;
  int L = __ldg(context_lens + b);
  L = L < 0 ? 0 : (L > max_len ? max_len : L);
  const int nreal = min(nq, next_n - gi * nq);
  const int vis = causal ? min(max(L - next_n + gi * nq + nreal, 0), L) : L;
  return (vis + 127) / 128;
}

// Plan of the fused call.  Lays the query groups end to end on a line, group u taking
// `cost` + (its visible key tiles) positions (prefix[u] = its start, prefix[units] = the
// line length S), and cuts the line into `slices` equal slices of Q = ceil(S / slices)
// positions.  When the longest group fills at most half a slice, whole groups balance
// well enough: mode kPlanGroups, with the groups listed longest first in `order` (by
// buckets of equal length).  Otherwise mode kPlanSlices: the group holding each slice's
// first position goes to ufirst, the groups whose tiles fall in more than one slice to
// `split`.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ context_lens, int B, int next_n,
                                                    int causal, int max_len, int nq, int ngroups, int slices,
                                                    int cost, int32_t* plan, int32_t* prefix, int32_t* ufirst,
                                                    int32_t* split, int32_t* order) {
  grid_launch_dependents();                 // the indexer's set-up may overlap this kernel
  constexpr int kBuckets = 4096;
  __shared__ int s_warp[32];
  __shared__ int s_carry, s_nsplit, s_max;
  __shared__ int s_hist[kBuckets];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int units = B * ngroups;
  if (tid == 0) {
    s_carry = 0;
    s_nsplit = 0;
    s_max = 0;
  }
  __syncthreads();
  // 1. prefix sums of the group weights; longest group
  int lmax = 0;
  for (int u0 = 0; u0 < units; u0 += 1024) {
    const int u = u0 + tid;
    const int tiles = u < units ? group_tiles(context_lens, u, ngroups, nq, next_n, causal, max_len) : 0;
    const int w = u < units ? tiles + cost : 0;
    lmax = max(lmax, tiles);
    int x = w;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
      const int v = s_warp[lane];
      int z = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, z, o);
        if (lane >= o) z += y;
      }
      s_warp[lane] = z - v;
    }
    __syncthreads();
    const int start = s_carry + s_warp[wid] + x - w;
    if (u < units) prefix[u] = start;
    __syncthreads();
    if (tid == 1023) s_carry = start + w;
    __syncthreads();
  }
  for (int o = 16; o > 0; o >>= 1) lmax = max(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
  if (lane == 0) atomicMax(&s_max, lmax);
  for (int i = tid; i < kBuckets; i += 1024) s_hist[i] = 0;
  __syncthreads();
  const int S = s_carry;
  const int mx = s_max;
  const int Q = S > 0 ? (S + slices - 1) / slices : 1;
  const int mode = (int64_t)2 * (mx + cost) <= Q ? kPlanGroups : kPlanSlices;
  if (tid == 0) prefix[units] = S;
  __syncthreads();
  if (mode == kPlanSlices) {
    // 2. first group of every slice; split groups
    for (int u = tid; u < units; u += 1024) {
      const int a0 = prefix[u], a1 = prefix[u + 1];
      for (int r = (a0 + Q - 1) / Q; r < slices && (int64_t)r * Q < a1; ++r) ufirst[r] = u;
      if (group_is_split(a0, a1, cost, Q)) {
        const int at = atomicAdd(&s_nsplit, 1);
        if (at < slices) split[at] = u;
      }
    }
  } else {
    // 2'. groups longest first: counting sort over length buckets
    const int per = (mx + kBuckets) / kBuckets;             // tiles per bucket (>= 1)
    for (int u = tid; u < units; u += 1024) {
      const int tiles = prefix[u + 1] - prefix[u] - cost;
      atomicAdd(&s_hist[kBuckets - 1 - tiles / per], 1);
    }
    __syncthreads();
    {
      int v[kBuckets / 1024], sum = 0;
#pragma unroll
      for (int i = 0; i < kBuckets / 1024; ++i) {
        v[i] = s_hist[tid * (kBuckets / 1024) + i];
        sum += v[i];
      }
      int incl = sum;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_warp[wid] = incl;
      __syncthreads();
      if (wid == 0) {
        const int w0 = s_warp[lane];
        int z = w0;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, z, o);
          if (lane >= o) z += y;
        }
        s_warp[lane] = z - w0;
      }
      __syncthreads();
      int acc = s_warp[wid] + incl - sum;
#pragma unroll
      for (int i = 0; i < kBuckets / 1024; ++i) {
        s_hist[tid * (kBuckets / 1024) + i] = acc;
        acc += v[i];
      }
    }
    __syncthreads();
    for (int u = tid; u < units; u += 1024) {
      const int tiles = prefix[u + 1] - prefix[u] - cost;
      order[atomicAdd(&s_hist[kBuckets - 1 - tiles / per], 1)] = u;
    }
  }
  __syncthreads();
  if (tid == 0) {
    plan[0] = Q;
    plan[1] = S;
    plan[2] = min(s_nsplit, slices);
    plan[3] = cost;
    plan[4] = mode;
    plan[5] = 0;                            // work counter (mode kPlanGroups)
    plan[6] = 0;
    plan[7] = 0;
    if (s_nsplit > slices) raise_error(DSA_DEVERR_OVERFLOW | (50u << 8));
  }
}

// =====================================================================================
// Host side
// =====================================================================================

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D map over rows of 128 elements (bf16 or byte), 128-byte swizzle, box = 128 bytes x box_rows.
bool make_map(CUtensorMap* m, const void* base, bool fp8, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {fp8 ? 128ull : 256ull};
  const cuuint32_t box[2] = {fp8 ? 128u : 64u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr size_t kSmemLimit = 232448;   // max dynamic shared memory per CTA (227 KB)
constexpr size_t kSmemHalf = 115712;    // two CTAs per SM (228 KB per SM, 1 KB reserved per CTA)
constexpr int64_t kSplitUnits = 1216;   // logits mode: fewer query groups than this: split key chunks

size_t smem_bytes(bool fp8, int nq, int stages, bool topk, int cap, int pow2, bool binned = false) {
  const size_t elt = fp8 ? 1 : 2;
  size_t s = 1024;                                    // alignment slack
  s += (size_t)nq * 64 * 128 * elt;                  // Q tile
  s += (size_t)stages * 128 * 128 * elt;             // key ring
  s += (size_t)(2 * stages + 16) * 8;                // barriers
  s += sizeof(EpiSmem<4>) + 16;
  if (topk) s += (size_t)nq * cap * 8;                                     // candidate buffers
  if (topk && binned) s += (size_t)(pow2 + kItemMaxBin) * 8 + kCutBins * 4;   // binned top k
  return s;
}

// FP4-key mode: `conv` padded E2M1 key tiles of 128 x 128 bytes, the E4M3 Q tile,
// `stages` FP4 stages of 128 x (64 + 4) bytes.
size_t smem_bytes_f4k(int nq, int stages, int conv, bool topk, int cap, int pow2, bool binned = false) {
  size_t s = 1024;
  s += (size_t)conv * 128 * 128;                     // padded key tiles
  s += (size_t)nq * 64 * 128;                        // E4M3 Q tile
  s += (size_t)stages * 128 * 68;                    // FP4 stages
  s += (size_t)((2 * stages + 16 + 2 * conv + 1) & ~1) * 8;   // barriers (an even count)
  s += sizeof(EpiSmem<4>) + 16;
  if (topk) s += (size_t)nq * cap * 8;                                     // candidate buffers
  if (topk && binned) s += (size_t)(pow2 + kItemMaxBin) * 8 + kCutBins * 4;   // binned top k
  return s;
}

}  // namespace

IndexerPlan plan_indexer(dsa_dtype dt, const dsa_queries& qs, int topk, bool wide) {
  IndexerPlan pl{};
  const bool fp8 = dt != DSA_BF16;                   // E4M3 queries
  const bool tk = topk > 0;
  pl.f4k = dt == DSA_E4M3_MXFP4K;
  pl.nq = qs.next_n == 1 ? 1 : (qs.next_n == 2 ? 2 : 4);
  if (pl.f4k && pl.nq > 2) pl.nq = 2;                // FP4 keys: <= 2 rows per item
  if (tk) {
    pl.pow2 = next_pow2(topk);
    // room for several tiles of inserts between cut-backs
    const int c0 = pl.pow2 > 2 * topk ? pl.pow2 : (topk + 1024 > 2 * topk ? topk + 1024 : 2 * topk);
    pl.cap = ((c0 + 255) / 256) * 256;
    if (pl.cap > 256 * kMaxPer) pl.cap = 256 * kMaxPer;
  }
  pl.ok = true;
  // One epilogue group (192 threads) for one or two query rows per item, with two CTAs
  // per SM where shared memory allows; otherwise (and for four rows) one CTA per SM
  // with two groups (320 threads).
  for (;;) {
    pl.eg = pl.nq <= 2 ? 1 : 2;
    int st = 4;
    while (st >= 2 && smem_bytes(fp8, pl.nq, st, tk, pl.cap, pl.pow2) > kSmemLimit) --st;
    if (st >= 2) {
      pl.stages = st;
      break;
    }
    if (pl.nq == 1) {
      pl.ok = false;
      return pl;
    }
    pl.nq >>= 1;
  }
  pl.ctas_per_sm = 1;
  if (pl.eg == 1) {
    int st = 4;
    while (st >= 2 && smem_bytes(fp8, pl.nq, st, tk, pl.cap, pl.pow2) > kSmemHalf) --st;
    if (st >= 2) {
      pl.stages = st;
      pl.ctas_per_sm = 2;
    }
  }
  if (pl.ctas_per_sm == 1 && pl.nq >= 2) pl.eg = 2;   // one CTA per SM: two groups take turns
  if (tk && (pl.cap < topk + 256 || pl.cap < pl.pow2)) pl.ok = false;
  pl.smem = smem_bytes(fp8, pl.nq, pl.stages, tk, pl.cap, pl.pow2);
  // Two epilogue groups check their buffers at every tile unless the buffers are wider than
  // k + 1024: with k + 512 + 512 c keys, every c-th tile (fewer cut-backs and group barriers).
  // The plan takes, in this order, k + 2048 keys at its depth, k + 1536 at its depth, then
  // the same at one pipeline stage less (two at least; not in the FP4-key mode); the
  // occupancy never changes.  Measured: FP8 chunked 9.41 -> 8.00 ms (k + 2048, every third
  // tile), bf16 prefill 2.87 -> 2.62 ms (k + 2048 at two stages), Pro decode MTP 0.170 ->
  // 0.164 ms (k + 1536 at four stages; k + 2048 at three was slower).
  auto widen = [&](auto smem_of) {
    pl.check_every = pl.eg == 1 ? 2 : 1;
    if (!tk || pl.eg != 2 || !wide) return;
    const size_t lim = pl.ctas_per_sm == 2 ? kSmemHalf : kSmemLimit;
    const int st0 = pl.stages, st_min = pl.f4k ? st0 : std::max(2, st0 - 1);
    for (int st = st0; st >= st_min; --st) {
      for (int extra = 2048; extra >= 1536; extra -= 512) {
        const int want = topk + extra;
        if (want > 256 * kMaxPer2) continue;
        const int cap2 = (want + 255) / 256 * 256;
        const int ci = (cap2 - topk - 512) / 512;
        if (cap2 <= pl.cap) {                  // the buffers are that wide already
          pl.check_every = std::max(1, (pl.cap - topk - 512) / 512);
          return;
        }
        const size_t sb = smem_of(cap2, st);
        if (sb <= lim) {
          pl.cap = cap2;
          pl.stages = st;
          pl.smem = sb;
          pl.check_every = ci;
          return;
        }
      }
    }
  };
  // the binned top k's gather buffer, only where it changes neither depth nor occupancy
  if (tk) {
    const size_t sb = smem_bytes(fp8, pl.nq, pl.stages, tk, pl.cap, pl.pow2, true);
    if (sb <= (pl.ctas_per_sm == 2 ? kSmemHalf : kSmemLimit)) {
      pl.binned = true;
      pl.smem = sb;
    }
  }
  widen([&](int c, int st) { return smem_bytes(fp8, pl.nq, st, tk, c, pl.pow2, pl.binned); });
  if (pl.f4k) {
    // one CTA per SM: two epilogue groups taking the tiles in turn, four converter warps,
    // a deep FP4 ring and as many padded key tiles (2..4) as shared memory holds
    pl.eg = 2;
    pl.ctas_per_sm = 1;
    pl.stages = 8;
    pl.conv_slots = 4;
    while (pl.conv_slots > 2 && smem_bytes_f4k(pl.nq, pl.stages, pl.conv_slots, tk, pl.cap, pl.pow2) > kSmemLimit)
      --pl.conv_slots;
    while (pl.stages > 2 && smem_bytes_f4k(pl.nq, pl.stages, pl.conv_slots, tk, pl.cap, pl.pow2) > kSmemLimit) --pl.stages;
    pl.smem = smem_bytes_f4k(pl.nq, pl.stages, pl.conv_slots, tk, pl.cap, pl.pow2);
    if (pl.smem > kSmemLimit) pl.ok = false;
    pl.binned = false;
    if (tk && smem_bytes_f4k(pl.nq, pl.stages, pl.conv_slots, tk, pl.cap, pl.pow2, true) <= kSmemLimit) {
      pl.binned = true;
      pl.smem = smem_bytes_f4k(pl.nq, pl.stages, pl.conv_slots, tk, pl.cap, pl.pow2, true);
    }
    widen([&](int c, int st) { return smem_bytes_f4k(pl.nq, st, pl.conv_slots, tk, c, pl.pow2, pl.binned); });
    // Each CTA holds all 512 TMEM columns (accumulators and scale cells): the request is
    // kept above half an SM's shared memory, so no second CTA is placed beside it.
    if (pl.smem <= kSmemHalf) pl.smem = kSmemHalf + 1024;
  }
  // as many accumulator buffers (up to 4) as TMEM holds for the CTAs sharing an SM, so
  // the MMAs can run ahead of an epilogue busy cutting its candidates back
  pl.nbuf_log2 = 2;
  while (pl.nbuf_log2 > 1 && pl.ctas_per_sm * next_pow2((pl.nq * 64) << pl.nbuf_log2) > 512) --pl.nbuf_log2;
  // FP4-key mode: the accumulators stay below column 256, the scale cells above it
  if (pl.f4k)
    while (pl.nbuf_log2 > 1 && ((pl.nq * 64) << pl.nbuf_log2) > 256) --pl.nbuf_log2;
  pl.ngroups = (qs.next_n + pl.nq - 1) / pl.nq;
  const int64_t units = (int64_t)qs.B * pl.ngroups;
  // logits mode: static chunks of the longest row, split when groups are few
  const int64_t full = ((int64_t)qs.max_context_len + 127) / 128 * 128;
  int64_t chunk = full;
  if (units < kSplitUnits) {
    const int64_t want = (full * units + 2431) / 2432;
    chunk = (want + 127) / 128 * 128;
    if (chunk < 2048) chunk = 2048;
    if (chunk > full) chunk = full;
  }
  if (chunk < 128) chunk = 128;
  pl.chunk = (int)chunk;
  pl.nchunks = (int)((qs.max_context_len + chunk - 1) / chunk);
  if (pl.nchunks < 1) pl.nchunks = 1;
  pl.items = units * pl.nchunks;
  // top-k mode: one slice of the plan's line per resident CTA; workspace = [plan header]
  // [prefix: units + 1][ufirst: slices][split: slices][order: units]
  // [partial lists: 2 per slice, cap keys per query row][their counts and thresholds]
  pl.slices = device_sm_count() * pl.ctas_per_sm;
  pl.cost = pl.nq == 4 ? 8 : 3;   // per-item cost in tile units: Q tile, drain, final ranking
  if (tk) {
    const int64_t max_tiles = ((int64_t)qs.max_context_len + 127) / 128;
    if (units * (max_tiles + pl.cost) >= (int64_t)INT32_MAX) pl.ok = false;   // line positions are int32
    size_t off = (size_t)kPlanHeader * 4;
    pl.prefix_off = off;
    off += (size_t)(units + 1) * 4;
    pl.ufirst_off = off;
    off += (size_t)pl.slices * 4;
    pl.split_off = off;
    off += (size_t)pl.slices * 4;
    pl.order_off = off;
    off += (size_t)units * 4;
    off = (off + 15) / 16 * 16;
    pl.partial_off = off;
    off += (size_t)pl.slices * 2 * pl.nq * pl.cap * 8;
    pl.meta_off = off;
    off += (size_t)pl.slices * 2 * pl.nq * 16;
    pl.ws_bytes = off;
    pl.items = units;
  }
  return pl;
}

cudaError_t launch_indexer(const IndexerArgs& a, const IndexerPlan& pl, cudaStream_t stream) {
  if (pl.items <= 0) return cudaSuccess;
  const bool paged = a.keys.block_table != nullptr;
  const int64_t T = (int64_t)a.qs.B * a.qs.next_n;
  CUtensorMap mq, mk;
  const uint32_t box_rows = paged ? (uint32_t)(a.keys.block_size < 128 ? a.keys.block_size : 128) : 128u;
  if (!make_map(&mq, a.q, a.fp8, (uint64_t)T * 64, (uint32_t)(pl.nq * 64))) return cudaErrorInvalidValue;
  if (pl.f4k) memset(&mk, 0, sizeof(mk));             // FP4 keys arrive by plain bulk copies
  else if (!make_map(&mk, a.keys.data, a.fp8, (uint64_t)a.keys.num_rows, box_rows)) return cudaErrorInvalidValue;
  IndexerParams prm{};
  prm.weights = a.weights;
  prm.q_scale = a.q_scale;
  prm.k_scale = a.keys.scale;
  prm.block_table = a.keys.block_table;
  prm.bt_stride = a.keys.bt_stride;
  prm.block_size = paged ? a.keys.block_size : 128;
  prm.num_blocks = paged ? a.keys.num_rows / a.keys.block_size : 0;
  prm.num_rows = a.keys.num_rows;
  prm.context_lens = a.qs.context_lens;
  prm.B = a.qs.B;
  prm.next_n = a.qs.next_n;
  prm.causal = a.qs.causal;
  prm.max_len = a.qs.max_context_len;
  prm.ngroups = pl.ngroups;
  prm.nchunks = pl.nchunks;
  prm.chunk = pl.chunk;
  prm.stages = pl.stages;
  prm.nbuf_log2 = pl.nbuf_log2;
  prm.kv_fp4 = pl.f4k ? static_cast<const uint8_t*>(a.keys.data) : nullptr;
  prm.kv_e8m0 = pl.f4k ? a.keys.scale_e8m0 : nullptr;
  prm.conv_slots = pl.conv_slots;
  prm.logits = a.logits;
  prm.ld = a.ld;
  prm.topk = a.topk;
  prm.cap = pl.cap;
  prm.pow2 = pl.pow2;
  prm.binned = pl.binned ? 1 : 0;
  prm.check_every = pl.check_every;
  prm.out_idx = a.out_idx;
  prm.out_val = a.out_val;
  const bool tk = a.topk > 0;
  int64_t grid = device_sm_count() * pl.ctas_per_sm;
  cudaError_t e;
  int32_t* split = nullptr;
  if (tk) {
    char* ws = static_cast<char*>(a.ws);
    int32_t* plan = reinterpret_cast<int32_t*>(ws);
    int32_t* prefix = reinterpret_cast<int32_t*>(ws + pl.prefix_off);
    int32_t* ufirst = reinterpret_cast<int32_t*>(ws + pl.ufirst_off);
    split = reinterpret_cast<int32_t*>(ws + pl.split_off);
    int32_t* order = reinterpret_cast<int32_t*>(ws + pl.order_off);
    prm.plan = plan;
    prm.prefix = prefix;
    prm.ufirst = ufirst;
    prm.order = order;
    prm.work = reinterpret_cast<uint32_t*>(plan + 5);
    prm.partial = reinterpret_cast<uint64_t*>(ws + pl.partial_off);
    prm.partial_meta = reinterpret_cast<uint64_t*>(ws + pl.meta_off);
    grid = pl.slices;
    plan_kernel<<<1, 1024, 0, stream>>>(a.qs.context_lens, a.qs.B, a.qs.next_n, a.qs.causal, a.qs.max_context_len,
                                        pl.nq, pl.ngroups, pl.slices, pl.cost, plan, prefix, ufirst, split, order);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else if (grid > pl.items) {
    grid = pl.items;
  }
  if (a.fp8)
    e = tk ? launch_indexer_fp8_topk(mq, mk, prm, pl, (int)grid, stream)
           : launch_indexer_fp8_logits(mq, mk, prm, pl, (int)grid, stream);
  else
    e = tk ? launch_indexer_bf16_topk(mq, mk, prm, pl, (int)grid, stream)
           : launch_indexer_bf16_logits(mq, mk, prm, pl, (int)grid, stream);
  if (e != cudaSuccess || !tk) return e;
  // groups cut by slice boundaries: rank their lists
  return launch_merge(prm.partial, prm.partial_meta, pl.cap, prm.plan, prm.prefix, split, pl.slices, pl.nq, a.qs,
                      a.topk, a.out_idx, a.out_val, stream);
}

DSA_DEFINE_TU_ERROR_ACCESSORS(indexer)

}  // namespace dsa
