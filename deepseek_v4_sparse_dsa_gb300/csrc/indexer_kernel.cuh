// The persistent tcgen05 indexer kernel (score, fused top-k) as a template; each
// indexer_<dtype>_<mode>.cu translation unit instantiates one (dtype, mode) pair so the
// variants compile in parallel.  Planning, the plan kernel and the launch sequence are
// in indexer.cu.
//
// DSA indexer score and fused top-k on tcgen05 tensor cores (sm_103a).
//
// Score (xkernels issue #27 "DSA indexer + attention: validate/provide gfx942 forward
// path", comment 2 "What shipped"):  logits[t, j] = sum_h w[t, h] * relu(q[t, h, :] . k[j, :]).
//
// Work item = (sequence b, a group of NQ query rows, a range of key tiles).  The
// contraction runs key-major: A = a tile of 128 keys x D (K-major, shared memory), B =
// the NQ*64 (query, head) rows of q x D, so the accumulator D[key, (query, head)] sits in
// tensor memory with one key per TMEM lane.  An epilogue thread owns one key and reduces
// its 64 head columns in registers: ReLU, weight and head sum need no cross-thread traffic.
//
// The kernel is persistent.  In top-k mode a one-CTA plan kernel first reads the actual
// context lengths and lays every query group's key tiles end to end, each group weighted
// by its tiles plus a fixed per-item cost.  When every group is short next to a CTA's
// share, CTAs take whole groups longest first through an atomic counter; otherwise CTA
// i takes the i-th of gridDim.x equal slices of that line: a group inside one slice is
// finished by one CTA, a group cut by slice boundaries leaves one unsorted candidate
// list per slice that the merge kernel (topk.cu) ranks.  (Logits mode, which has no
// workspace, walks fixed chunks with a static stride.)  Warp roles (64 + 128 * EG
// threads):
//   warp 0     producer: walks its items, publishes their descriptors, loads each item's
//              Q tile and streams key tiles into an S-stage ring with TMA (paged keys:
//              one box per page, block ids read from a shared-memory window the whole
//              warp refills); it runs ahead of the other roles across item boundaries
//   warp 1     TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2..  EG epilogue groups of 4 warps; global tile T uses TMEM buffer T % NB and
//              epilogue group T % EG
//   (FP4 keys) four converter warps after them: padded E2M1 tiles and TMEM scale cells
//              for the block-scaled MMA
// Epilogue: tcgen05.ld of each query's 64 head sums, fp32 ReLU * weight head sum in a
// fixed order, then a store of the score row (logits mode) or an insert into a per-query
// candidate buffer in shared memory (top-k mode) that a histogram cut brings back to a
// superset of the top-k whenever it fills.  Unsplit groups get each row's top k here, by
// value bins (engine_topk_binned), the whole epilogue on one row after another.
//
// Every wait is bounded (see common.cuh); a timeout abandons the work, flags
// DSA_DEVERR_TIMEOUT, waits for this CTA's own copies and MMAs, frees TMEM and returns.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace dsa {

struct IndexerParams {
  const float* weights;
  const float* q_scale;
  const float* k_scale;
  const int32_t* block_table;
  int64_t bt_stride;
  int64_t num_blocks;       // pool blocks (paged)
  int64_t num_rows;         // key rows in the pool / contiguous key array
  const int32_t* context_lens;
  float* logits;
  int64_t ld;
  int32_t* out_idx;
  float* out_val;
  uint64_t* partial;        // [slice][head, tail][NQ][cap] candidate keys of split groups' pieces
  uint64_t* partial_meta;   // [slice][head, tail][NQ][2]: candidate count, piece threshold
  const int32_t* plan;      // top-k mode: plan header (slice length, total, split count, item cost)
  const int32_t* prefix;    // top-k mode: [units + 1] start of each query group on the line
  const int32_t* ufirst;    // top-k mode: [slices] the group holding each slice's first position
  const int32_t* order;     // top-k mode: [units] groups longest first (plan mode kPlanGroups)
  uint32_t* work;           // top-k mode: work counter in the plan header (plan mode kPlanGroups)
  int32_t block_size;
  int32_t B, next_n, causal, max_len;
  int32_t ngroups, nchunks, chunk;  // static schedule (logits mode)
  int32_t topk, cap, pow2, stages;
  int32_t nbuf_log2;        // log2 of the TMEM accumulator buffers (1 or 2)
  int32_t binned;           // top-k mode: whole groups ranked by value bins (gather buffer present)
  int32_t check_every;      // top-k mode: tiles between buffer checks (1 or 2)
  // FP4-key mode: keys read from the paged mxfp4 cache (nibble rows of 64 bytes, E8M0
  // rows of 4 bytes), repacked on chip for the block-scaled MMA by the converter warps
  const uint8_t* kv_fp4;
  const uint8_t* kv_e8m0;
  int32_t conv_slots;       // padded E2M1 key tiles in flight
};

constexpr int kMaxPer = 10;        // candidate capacity per query <= 256 * kMaxPer
constexpr int kMaxPer2 = 12;       // two epilogue groups: up to 256 * kMaxPer2 (wider buffers)
constexpr uint32_t kItemMaxBin = 512;   // binned top k of a whole group: largest bin gathered

struct ItemInfo {
  int32_t valid, b, g, L, nreal, vis_max;
  int32_t ks, ke, ntiles;   // keys [ks, ke) in ntiles tiles of 128
  int32_t t0, chunk;        // first query row; chunk length (logits mode: masked tail)
  int32_t split, slot;      // top-k mode: group cut by slice boundaries; its list slot
  int32_t vis[4];
};

constexpr int kPageWindow = 256;    // block-table entries the producer keeps in shared memory

template <int NQ>
struct EpiSmem {
  int32_t pages[kPageWindow];
  float w[2][NQ][64];
  ItemInfo info[2];
  uint32_t tmem_base;
  int abort;
  int stop;
  int last;
  int cstop;                // FP4-key mode: the converters' own stop decision
  uint32_t cnt[4];
  uint64_t thr[4];
  EngineScratch esc;
  alignas(16) uint32_t bins[kCutBins];
};

// Two fp32 fused multiply-adds in one instruction (each lane rounded as fmaf).
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}

// sum_h w[h] * relu(s[h]) in a fixed order: four interleaved partial sums p_r over
// h = r (mod 4), then (p0 + p1) + (p2 + p3); pairs (p0, p1) and (p2, p3) advance with
// one two-lane FMA each.
__device__ __forceinline__ float head_sum(const uint32_t (&s)[64], const float* w) {
  uint64_t a01 = 0ull, a23 = 0ull;
#pragma unroll
  for (int h = 0; h < 64; h += 4) {
    const float4 wv = *reinterpret_cast<const float4*>(w + h);
    a01 = fma2(pack2(wv.x, wv.y),
               pack2(fmaxf(__uint_as_float(s[h + 0]), 0.f), fmaxf(__uint_as_float(s[h + 1]), 0.f)), a01);
    a23 = fma2(pack2(wv.z, wv.w),
               pack2(fmaxf(__uint_as_float(s[h + 2]), 0.f), fmaxf(__uint_as_float(s[h + 3]), 0.f)), a23);
  }
  const float a0 = __uint_as_float((uint32_t)a01), a1 = __uint_as_float((uint32_t)(a01 >> 32));
  const float a2 = __uint_as_float((uint32_t)a23), a3 = __uint_as_float((uint32_t)(a23 >> 32));
  return (a0 + a1) + (a2 + a3);
}

// Head sums of the NQ query rows of one key (this thread's TMEM lane) from the
// accumulator columns at `tcol`: the load of row q + 1 overlaps the sum of row q.
template <int NQ>
__device__ __forceinline__ void head_sums(uint32_t tcol, const float* wq, float (&v)[NQ]) {
  uint32_t ra[64], rb[64];
  tmem_ld64_issue(tcol, ra);
  tmem_ld64_wait(ra);
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (q & 1) {
      if (q + 1 < NQ) tmem_ld64_issue(tcol + (uint32_t)((q + 1) * 64), ra);
      v[q] = head_sum(rb, wq + q * 64);
      if (q + 1 < NQ) tmem_ld64_wait(ra);
    } else {
      if (q + 1 < NQ) tmem_ld64_issue(tcol + (uint32_t)((q + 1) * 64), rb);
      v[q] = head_sum(ra, wq + q * 64);
      if (q + 1 < NQ) tmem_ld64_wait(rb);
    }
  }
}

// Query group u = b * ngroups + gi: its sequence, rows and visible key counts.
template <int NQ>
__device__ void decode_group(const IndexerParams& p, int u, ItemInfo& it) {
  const int b = u / p.ngroups;
  const int gi = u - b * p.ngroups;
  int L = __ldg(p.context_lens + b);
  if (L < 0 || L > p.max_len) {
    raise_error(DSA_DEVERR_INDEX);
    L = L < 0 ? 0 : p.max_len;
  }
  const int i0 = gi * NQ;
  const int nreal = min(NQ, p.next_n - i0);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    int v = 0;
    if (q < nreal) v = p.causal ? min(max(L - p.next_n + i0 + q + 1, 0), L) : L;
    it.vis[q] = v;
  }
  it.valid = 1;
  it.b = b;
  it.g = gi;
  it.L = L;
  it.nreal = nreal;
  it.vis_max = p.causal ? min(max(L - p.next_n + i0 + nreal, 0), L) : L;
  it.t0 = b * p.next_n + i0;
  it.split = 0;
  it.slot = 0;
  it.chunk = 0;
}

// Logits mode: group u, fixed key chunk c.
template <int NQ>
__device__ void decode_chunk_item(const IndexerParams& p, int u, int c, ItemInfo& it) {
  decode_group<NQ>(p, u, it);
  const int ks = c * p.chunk;
  const int ke = min(ks + p.chunk, it.vis_max);
  it.ks = ks;
  it.ke = ke > ks ? ke : ks;
  it.ntiles = ke > ks ? (ke - ks + 127) / 128 : 0;
  it.chunk = p.chunk;
}

// Top-k mode: the next item of slice [r0, r1) of the plan's line, walking groups from
// *u on.  A group with line span [a0, a1) spends its first `cost` positions on its fixed
// item cost and then has one position per key tile; a group without tiles belongs to
// the slice that holds its position a0.  Returns false when the slice holds no more.
template <int NQ>
__device__ bool next_slice_item(const IndexerParams& p, int slice, int r0, int r1, int Q, int cost, int units,
                                int* u, ItemInfo& it) {
  while (*u < units) {
    const int g = *u;
    const int a0 = __ldcg(p.prefix + g), a1 = __ldcg(p.prefix + g + 1);
    if (a0 >= r1) return false;
    *u = g + 1;
    const int tiles = a1 - a0 - cost;
    if (tiles <= 0) {
      if (a0 / Q != slice) continue;
      decode_group<NQ>(p, g, it);
      it.ks = it.ke = it.ntiles = 0;
      return true;
    }
    const int rs = a0 + cost;
    const int lo = max(r0, rs), hi = min(r1, a1);
    if (lo >= hi) continue;
    decode_group<NQ>(p, g, it);
    it.ks = (lo - rs) * 128;
    it.ke = min((hi - rs) * 128, it.vis_max);
    it.ntiles = hi - lo;
    it.split = group_is_split(a0, a1, cost, Q) ? 1 : 0;
    it.slot = split_slot(slice, a0, cost, Q);
    return true;
  }
  return false;
}

// E8M0 scale cells for the tensor cores: a byte 0xFF (scale 0 here, NaN there) becomes 127.
__device__ __forceinline__ uint32_t e8m0_ff_to_one(uint32_t w) {
  return w ^ (__vcmpeq4(w, 0xFFFFFFFFu) & 0x80808080u);
}

template <bool kFP8, int NQ, bool kTopk, int EG, bool kF4K>
__global__ void __launch_bounds__(64 + 128 * EG + (kF4K ? 128 : 0), (EG == 1 && !kF4K) ? 2 : 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const IndexerParams p) {
  // kF4K: E4M3 queries against mxfp4 keys, contracted by the block-scaled MMA: the key
  // codes in the padded E2M1 layout, their E8M0 scales in tensor memory, the E4M3 Q tile
  // as loaded with scale 1.
  static_assert(!kF4K || kFP8, "FP4-key mode: E4M3 queries");
  constexpr bool kMmaFP8 = kFP8 && !kF4K;          // E4M3 x E4M3 contraction
  constexpr bool kKeyScale = kFP8 && !kF4K;        // per-key fp32 scale (E4M3 keys)
  constexpr int N = NQ * 64;                       // MMA N: (query, head) rows
  constexpr int ELT = kFP8 ? 1 : 2;                // bytes per element as stored in HBM
  constexpr int KCH = kMmaFP8 ? 1 : 2;             // 128-byte K chunks per row in the MMA operands
  constexpr uint32_t Q_CHUNK = N * 128;            // bytes of one K chunk of the Q tile
  constexpr uint32_t Q_BYTES = Q_CHUNK * KCH;
  constexpr uint32_t K_CHUNK = 128 * 128;          // 128 keys x 128 bytes
  constexpr uint32_t K_BYTES = K_CHUNK * KCH;
  constexpr int KSTEPS = KCH * 4;                  // 32 bytes of K per MMA
  constexpr uint32_t F4_BYTES = 128 * 64 + 128 * 4;   // FP4-key stage: nibble rows, then E8M0 rows
  constexpr uint32_t KT_BYTES = kF4K ? K_CHUNK : K_BYTES;   // kF4K: a padded E2M1 tile, 128 B per key
  constexpr uint32_t QS_BYTES = kF4K ? 0u : Q_BYTES;        // kF4K: the E4M3 Q tile is the operand as loaded
  const int NBL = p.nbuf_log2;                     // NB = 2^NBL accumulator buffers in TMEM
  const int NBM = (1 << NBL) - 1;
  // kF4K: accumulators in columns [0, 256), then the scale cells: 8 columns of the queries'
  // scale bytes (all 127: scale 1), 4 columns of key scale bytes per converted tile
  constexpr uint32_t SFB_COL = 256, SFA_COL = 264;
  const uint32_t TMEM_COLS = kF4K ? 512u : ((N << NBL) < 32) ? 32u : (uint32_t)next_pow2(N << NBL);
  constexpr uint32_t IDESC = kMmaFP8 ? idesc_e4m3(128, N) : idesc_bf16(128, N);

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment by pointer arithmetic on the shared array (not through an
  // integer), so the compiler keeps every access below in the shared window
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = p.stages;
  const int CR = kF4K ? p.conv_slots : 0;
  // layout: Q tile (MMA operand; none in kF4K) | key stages (TMA) or padded key tiles [CR]
  //         (kF4K) | kF4K: E4M3 Q tile, FP4 stages [S] | barriers | epilogue state
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + QS_BYTES;                        // S stages (kF4K: CR padded tiles)
  uint8_t* q8_s = k_s + (size_t)(kF4K ? CR : S) * KT_BYTES;  // kF4K: the E4M3 Q tile as loaded
  uint8_t* f4_s = q8_s + (kF4K ? Q_CHUNK : 0);           // kF4K: S stages of F4_BYTES
  uint64_t* bars = reinterpret_cast<uint64_t*>(f4_s + (kF4K ? (size_t)S * F4_BYTES : 0));
  // full[S] | empty[S] | tfull[4] | tempty[4] | qfull | qempty | ifull[2] | iempty[2] | mmadone | tmemfree
  // | kF4K: cfull[CR] | cfree[CR]
  const int NBARS = (2 * S + 16 + (kF4K ? 2 * CR : 0) + 1) & ~1;   // even: es stays 16-byte aligned
  EpiSmem<NQ>* es = reinterpret_cast<EpiSmem<NQ>*>(bars + NBARS);
  uint64_t* ebuf = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(es) + (sizeof(EpiSmem<NQ>) + 15) / 16 * 16);
  // top-k mode: the candidate buffers [NQ][cap], then (p.binned) the gather buffer of the
  // binned top k (pow2 + kItemMaxBin keys) and its bin starts (kCutBins words)
  uint64_t* tbuf = ebuf + (size_t)NQ * p.cap;
  uint32_t* tstart = reinterpret_cast<uint32_t*>(tbuf + p.pow2 + kItemMaxBin);

  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
  const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 4);
  const uint32_t qfull = smem_u32(bars + 2 * S + 8), qempty = smem_u32(bars + 2 * S + 9);
  const uint32_t ifull0 = smem_u32(bars + 2 * S + 10), iempty0 = smem_u32(bars + 2 * S + 12);
  const uint32_t mmadone = smem_u32(bars + 2 * S + 14);
  const uint32_t tmemfree = smem_u32(bars + 2 * S + 15);   // every epilogue warp is done with TMEM
  const uint32_t cfull0 = smem_u32(bars + 2 * S + 16), cfree0 = cfull0 + 8u * (uint32_t)CR;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned long long limit = wait_limit_ns();
  volatile int* abort_flag = &es->abort;
  const bool paged = p.block_table != nullptr;
  const int bs = p.block_size;

  // ---- setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kF4K ? 4 : 1);   // kF4K: the converter warps free FP4 stages
    }
    for (int c = 0; c < CR; ++c) {
      mbar_init(cfull0 + 8 * c, 4);              // the 4 converter warps wrote the tile
      mbar_init(cfree0 + 8 * c, 1);              // the MMAs that read it are done
    }
    for (int a = 0; a < 4; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);          // the 4 warps of the group that read the tile
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(ifull0 + 8 * a, 1);
      mbar_init(iempty0 + 8 * a, 1 + 4 * EG + (kF4K ? 4 : 0));
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, 1);
    mbar_init(mmadone, 1);
    mbar_init(tmemfree, 4 * EG + (kF4K ? 4 : 0));   // kF4K: the converters write scale cells
    es->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&es->tmem_base), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = es->tmem_base;

  if (warp == 0) {
    // ============================ producer (whole warp) ============================
    // Lane 0 owns the barriers and issues every copy; the other lanes help load the
    // block table into a shared window so no copy waits on a dependent global load.
    // Top-k mode: this CTA's slice [r0, r1) of the plan's line (the plan kernel may
    // still be running: wait for it first).  Logits mode: items blockIdx.x + k * grid.
    const int units = p.B * p.ngroups;
    int Q = 1, cost = 0, r0 = 0, r1 = 0, ucur = units, mode = kPlanSlices;
    int next = (int)blockIdx.x;
    const int chunk_items = units * p.nchunks;
    if (p.plan) {
      grid_dependency_wait();
      Q = __ldcg(p.plan);
      const int S = __ldcg(p.plan + 1);
      cost = __ldcg(p.plan + 3);
      mode = __ldcg(p.plan + 4);
      r0 = (int)blockIdx.x * Q;
      r1 = min(r0 + Q, S);
      if (mode == kPlanSlices && r0 < S) ucur = __ldcg(p.ufirst + blockIdx.x);
    }
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      if (!kF4K) tma_prefetch_desc(&tm_k);
      if (p.plan && mode == kPlanGroups) next = (int)atomicAdd(p.work, 1u);   // one item ahead
    }
    int tiles_issued = 0, items_issued = 0;
    int s_run = 0;                                          // stage of the next tile (tiles_issued % S)
    uint32_t ph_run = 0;                                    // its ring pass parity
    const int bsl = (bs & (bs - 1)) == 0 ? __ffs(bs) - 1 : -1;   // log2(block size), or -1
    int last_issue[8];
    for (int s = 0; s < 8; ++s) last_issue[s] = -1;
    bool ok = true;
    for (int n = 0;; ++n) {
      const int slot = n & 1;
      int have = 0;
      if (lane == 0) {
        ok = mbar_wait(iempty0 + 8 * slot, ((uint32_t)(n >> 1) & 1u) ^ 1u, limit, abort_flag);
        ItemInfo it;
        it.valid = 0;
        if (ok) {
          if (p.plan && mode == kPlanSlices) {
            have = next_slice_item<NQ>(p, (int)blockIdx.x, r0, r1, Q, cost, units, &ucur, it) ? 1 : 0;
          } else if (p.plan) {
            if (next < units) {
              const int g = __ldcg(p.order + next);
              next = (int)atomicAdd(p.work, 1u);
              decode_group<NQ>(p, g, it);
              it.ks = 0;
              it.ke = it.vis_max;
              it.ntiles = (it.vis_max + 127) / 128;
              have = 1;
            }
          } else if (next < chunk_items) {
            const int u = next / p.nchunks;
            decode_chunk_item<NQ>(p, u, next - u * p.nchunks, it);
            next += (int)gridDim.x;
            have = 1;
          }
        }
        es->info[slot] = it;
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      have = __shfl_sync(0xFFFFFFFFu, have, 0);
      if (!ok) break;
      if (!have) {
        if (lane == 0) mbar_arrive(ifull0 + 8 * slot);      // end-of-work descriptor
        break;
      }
      __syncwarp();
      const ItemInfo it = es->info[slot];
      // this item's Q tile, once the previous item's MMAs are done with the last one
      if (lane == 0) {
        ok = mbar_wait(qempty, ((uint32_t)n & 1u) ^ 1u, limit, abort_flag);
        if (ok) {
          if (kF4K) {                           // the E4M3 tile, the MMAs' B operand as loaded
            mbar_arrive_expect_tx(qfull, Q_CHUNK);
            tma_load_2d(smem_u32(q8_s), &tm_q, qfull, 0, it.t0 * 64);
          } else {
            mbar_arrive_expect_tx(qfull, Q_BYTES);
            for (int kc = 0; kc < KCH; ++kc)
              tma_load_2d(smem_u32(q_s + kc * Q_CHUNK), &tm_q, qfull, kc * (128 / ELT), it.t0 * 64);
          }
          ++items_issued;
          mbar_arrive(ifull0 + 8 * slot);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      // its key tiles
      const int ke = it.ke;
      int win0 = -1;                                        // first page held in the window
      for (int i = 0; i < it.ntiles; ++i) {
        const int T = tiles_issued + i;
        const int s = s_run;                                // T % S
        const int j0 = it.ks + i * 128;                     // a multiple of 128
        const int jend = min(j0 + 128, ke);
        int pg0 = 0, pg1 = 0;
        if (paged) {
          pg0 = bsl >= 0 ? j0 >> bsl : j0 / bs;
          pg1 = bs >= 128 ? pg0 : (jend - 1) >> bsl;
          if (win0 < 0 || pg1 >= win0 + kPageWindow) {
            __syncwarp();
            win0 = pg0;
            const int pend = (ke - 1) / bs;
            for (int e = lane; e < kPageWindow; e += 32) {
              const int pg = win0 + e;
              int32_t blk = -1;
              if (pg <= pend && pg < p.bt_stride) blk = __ldg(p.block_table + (int64_t)it.b * p.bt_stride + pg);
              es->pages[e] = blk;
            }
            __syncwarp();
          }
        }
        // Block size < 128 (a power of two dividing 128): lane k resolves page pg0 + k of
        // the tile (at most 16) while lane 0 waits for the stage, then issues its copies.
        const bool small_pages = paged && bs < 128;
        int64_t myblk = -1;
        const bool mine = small_pages && pg0 + lane <= pg1;
        if (mine) myblk = es->pages[pg0 + lane - win0];
        if (lane == 0) ok = mbar_wait(empty0 + 8 * s, ph_run ^ 1u, limit, abort_flag);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const uint32_t stage = smem_u32(k_s + (size_t)s * K_BYTES);
        const uint32_t fb = full0 + 8 * s;
        const uint32_t f4 = kF4K ? smem_u32(f4_s + (size_t)s * F4_BYTES) : 0u;
        if (small_pages) {
          const bool good = mine && myblk >= 0 && myblk < p.num_blocks;
          const uint32_t gm = __ballot_sync(0xFFFFFFFFu, good);
          const uint32_t bm = __ballot_sync(0xFFFFFFFFu, mine && !good);
          if (lane == 0) {
            if (bm) raise_error(DSA_DEVERR_INDEX);
            // nibble and E8M0 rows (kF4K), or the page's rows of every K chunk
            const uint32_t per_page = kF4K ? (uint32_t)bs * 68u : (uint32_t)bs * 128u * KCH;
            mbar_arrive_expect_tx(fb, (uint32_t)__popc(gm) * per_page);
          }
          __syncwarp();
          if (good) {
            const uint32_t at = (uint32_t)lane * (uint32_t)bs;     // the page's first row in the tile
            const int64_t row = myblk * bs;
            if constexpr (kF4K) {
              // plain bulk copies: 64 + 4 bytes per key, every source and size a multiple of 16 bytes
              bulk_load(f4 + at * 64u, p.kv_fp4 + (size_t)row * 64, (uint32_t)bs * 64u, fb);
              bulk_load(f4 + 8192u + at * 4u, p.kv_e8m0 + (size_t)row * 4, (uint32_t)bs * 4u, fb);
            } else {
              for (int kc = 0; kc < KCH; ++kc)
                tma_load_2d(stage + at * 128u + kc * K_CHUNK, &tm_k, fb, kc * (128 / ELT), (int32_t)row);
            }
          }
        } else if (lane == 0) {
          if constexpr (kF4K) {
            if (!paged) {
              const int rows = (int)max((int64_t)0, min((int64_t)128, p.num_rows - j0));
              mbar_arrive_expect_tx(fb, (uint32_t)rows * 68u);
              if (rows > 0) {
                bulk_load(f4, p.kv_fp4 + (size_t)j0 * 64, (uint32_t)rows * 64u, fb);
                bulk_load(f4 + 8192u, p.kv_e8m0 + (size_t)j0 * 4, (uint32_t)rows * 4u, fb);
              }
            } else {                                        // one page of >= 128 rows
              const int64_t blk = es->pages[pg0 - win0];
              if (blk >= 0 && blk < p.num_blocks) {
                mbar_arrive_expect_tx(fb, 128u * 68u);
                const int64_t row = blk * bs + (j0 % bs);
                bulk_load(f4, p.kv_fp4 + (size_t)row * 64, 128u * 64u, fb);
                bulk_load(f4 + 8192u, p.kv_e8m0 + (size_t)row * 4, 128u * 4u, fb);
              } else {
                raise_error(DSA_DEVERR_INDEX);
                mbar_arrive_expect_tx(fb, 0);
              }
            }
          } else if (!paged) {
            mbar_arrive_expect_tx(fb, K_BYTES);
            for (int kc = 0; kc < KCH; ++kc)
              tma_load_2d(stage + kc * K_CHUNK, &tm_k, fb, kc * (128 / ELT), j0);
          } else {                                          // one page of >= 128 rows
            const int64_t blk = es->pages[pg0 - win0];
            if (blk >= 0 && blk < p.num_blocks) {
              mbar_arrive_expect_tx(fb, K_BYTES);
              const int32_t row = (int32_t)(blk * bs + (j0 % bs));
              for (int kc = 0; kc < KCH; ++kc)
                tma_load_2d(stage + kc * K_CHUNK, &tm_k, fb, kc * (128 / ELT), row);
            } else {
              raise_error(DSA_DEVERR_INDEX);
              mbar_arrive_expect_tx(fb, 0);
            }
          }
        }
        if (lane == 0) last_issue[s] = T;
        if (++s_run == S) {
          s_run = 0;
          ph_run ^= 1u;
        }
      }
      if (!ok) break;
      tiles_issued += it.ntiles;
    }
    if (lane == 0) {
      grid_launch_dependents();             // every copy is issued: the merge may start launching
      if (!ok) {
        raise_error(DSA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // Own copies must land before this CTA can exit (matters only after an abort).
      if (items_issued > 0) mbar_wait(qfull, (uint32_t)(items_issued - 1) & 1u, kCleanupWaitNs, nullptr);
      for (int s = 0; s < S && s < 8; ++s)
        if (last_issue[s] >= 0) mbar_wait(full0 + 8 * s, (uint32_t)(last_issue[s] / S) & 1u, kCleanupWaitNs, nullptr);
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      int T = 0;
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int slot = n & 1;
        if (!(ok = mbar_wait(ifull0 + 8 * slot, (uint32_t)(n >> 1) & 1u, limit, abort_flag))) break;
        const ItemInfo it = es->info[slot];
        if (!it.valid) break;
        // the Q tile, loaded by TMA
        if (!(ok = mbar_wait(qfull, (uint32_t)n & 1u, limit, abort_flag))) break;
        const uint32_t qbase = smem_u32(kF4K ? q8_s : q_s);
        for (int i = 0; i < it.ntiles; ++i, ++T) {
          const int s = kF4K ? T % CR : T % S;      // key stage, or (kF4K) padded key tile
          const int a = T & NBM;
          const uint32_t kready = kF4K ? cfull0 + 8 * s : full0 + 8 * s;
          const uint32_t kphase = (uint32_t)(kF4K ? T / CR : T / S) & 1u;
          ok = mbar_wait(kready, kphase, limit, abort_flag) &&
               mbar_wait(tempty0 + 8 * a, ((uint32_t)(T >> NBL) & 1u) ^ 1u, limit, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t stage = smem_u32(k_s + (size_t)s * KT_BYTES);
          const uint32_t d = tmem_base + (uint32_t)(a * N);
          if constexpr (kF4K) {
            // four K steps of 32: E2M1 keys (scale byte kk of the tile's cells) x E4M3 queries
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_mx(d, smem_desc_sw128(stage + (uint32_t)kk * 32u), smem_desc_sw128(qbase + (uint32_t)kk * 32u),
                     idesc_mx_e2m1_e4m3(128, N, (uint32_t)kk, (uint32_t)kk), tmem_base + SFA_COL + 4u * (uint32_t)s,
                     tmem_base + SFB_COL, kk > 0 ? 1u : 0u);
          } else
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            const uint32_t off = (uint32_t)(kk & 3) * 32u;   // 16 bf16 / 32 E4M3 along K
            const uint64_t adesc = smem_desc_sw128(stage + (uint32_t)(kk >> 2) * K_CHUNK + off);
            const uint64_t bdesc = smem_desc_sw128(qbase + (uint32_t)(kk >> 2) * Q_CHUNK + off);
            if (kMmaFP8)
              mma_e4m3(d, adesc, bdesc, IDESC, kk > 0 ? 1u : 0u);
            else
              mma_bf16(d, adesc, bdesc, IDESC, kk > 0 ? 1u : 0u);
          }
          mma_commit(kF4K ? cfree0 + 8 * s : empty0 + 8 * s);
          mma_commit(tfull0 + 8 * a);
        }
        if (!ok) break;
        mma_commit(qempty);                 // the Q tile is free once this item's MMAs are done
        mbar_arrive(iempty0 + 8 * slot);
      }
      if (!ok) {
        raise_error(DSA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // Every MMA issued so far must finish, and every epilogue warp must be done
      // reading, before TMEM is released.
      mma_commit(mmadone);
      mbar_wait(mmadone, 0, kCleanupWaitNs, nullptr);
      mbar_wait(tmemfree, 0, kCleanupWaitNs, nullptr);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  } else if (!kF4K || warp < 2 + 4 * EG) {
    // ============================ epilogue ============================
    // EG groups of 4 warps take the tiles in turn (global tile T goes to group T % EG);
    // all NT threads share the per-row candidate buffers and cut them back together.
    constexpr int NT = 128 * EG;
    constexpr int MAXPER = EG == 2 ? kMaxPer2 : kMaxPer * 2 / EG;     // candidate slots per thread in a cut-back
    const int et = threadIdx.x - 64;             // 0..NT-1
    const int grp = (warp - 2) >> 2;
    const int ew = warp - 2;                     // epilogue warp 0..4*EG-1
    const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;         // key row within the tile
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const int cap = p.cap;
    int T0 = 0;                                  // global index of the item's first tile
    for (int n = 0;; ++n) {
      const int slot = n & 1;
      bool ok = (lane == 0) ? mbar_wait(ifull0 + 8 * slot, (uint32_t)(n >> 1) & 1u, limit, abort_flag) : true;
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok && lane == 0) {
        raise_error(DSA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // One thread decides for all epilogue warps between two barriers (the abort flag
      // may change at any time); an expired wait means the producer is gone: stop as on
      // the end-of-work descriptor.
      group_sync<NT>();
      if (et == 0) es->stop = (*abort_flag != 0) || !es->info[slot].valid;
      group_sync<NT>();
      if (es->stop) break;
      const ItemInfo it = es->info[slot];
      // per-item head weights (q scale folded in for E4M3)
      for (int e = et; e < NQ * 64; e += NT) {
        const int q = e >> 6, h = e & 63;
        float w = 0.f;
        if (q < it.nreal) {
          const int64_t o = (int64_t)(it.t0 + q) * 64 + h;
          w = __ldg(p.weights + o);
          if (kFP8) w *= __ldg(p.q_scale + o);
        }
        es->w[slot][q][h] = w;
      }
      if (kTopk && et < NQ) {
        es->cnt[et] = 0;
        es->thr[et] = 0;
      }
      group_sync<NT>();
      const float* wq = &es->w[slot][0][0];
      const int niter = (it.ntiles + EG - 1) / EG;
      const int first = ((grp - T0) % EG + EG) % EG;   // this group's first local tile
      // Block id of this thread's key in local tile i (-1: past the row or the table).
      // Read one tile ahead so the load overlaps the wait for the accumulator.
      auto page_of = [&](int i) -> int64_t {
        const int jj = it.ks + i * 128 + row;
        const int64_t pg = jj / bs;
        return (jj < it.L && pg < p.bt_stride) ? (int64_t)__ldg(p.block_table + (int64_t)it.b * p.bt_stride + pg)
                                               : (int64_t)-1;
      };
      int64_t blk_next = (paged && first < it.ntiles) ? page_of(first) : -1;
      float ks_next = 1.f;                      // contiguous E4M3 keys: scale of the next tile's key
      if (kKeyScale && !paged && first < it.ntiles && it.ks + first * 128 + row < p.num_rows)
        ks_next = __ldg(p.k_scale + it.ks + first * 128 + row);
      for (int m = 0; m < niter; ++m) {
        // The buffers are checked every CI tiles (one barrier per check), leaving room for
        // CI tiles of appends per group: every second tile for one group; for two groups,
        // every (cap - k - 512) / 512 tiles where the plan gave them wider buffers, else at
        // every tile.
        const int CI = p.check_every;
        if (kTopk && m % CI == 0) {
          group_sync<NT>();
#pragma unroll 1
          for (int q = 0; q < NQ; ++q) {
            const uint32_t cn = min(es->cnt[q], (uint32_t)cap);   // (a count past cap only after
            if (cn > (uint32_t)(cap - 128 * EG * CI)) {              //  a flagged overflow)
              // cut back to a superset of the top-k; exactly only if the histogram
              // cannot free enough room
              uint64_t* buf = ebuf + (size_t)q * cap;
              const uint32_t room = (uint32_t)min((cap + p.topk) / 2, cap - 256 * EG * CI);
              uint64_t thr = engine_cut_approx<NT, MAXPER>(buf, &es->cnt[q], (int)cn, p.topk, room, es->bins,
                                                           &es->esc, et);
              if (thr == 0ull) {
                thr = engine_select<NT>(buf, (int)cn, p.topk, &es->esc, et);
                engine_compact<NT, MAXPER>(buf, &es->cnt[q], (int)cn, thr, &es->esc, et);
              }
              if (et == 0 && thr > es->thr[q]) es->thr[q] = thr;
              group_sync<NT>();
            }
          }
        }
        const int i = EG * m + first;
        if (i >= it.ntiles) continue;
        const int T = T0 + i;
        const int a = T & NBM;
        const int j = it.ks + i * 128 + row;
        bool valid = true;
        float kscale = 1.f;
        if (paged) {
          const int64_t blk = blk_next;
          if (i + EG < it.ntiles) blk_next = page_of(i + EG);
          valid = blk >= 0 && blk < p.num_blocks;
          if (kKeyScale && valid) kscale = __ldg(p.k_scale + blk * bs + (j % bs));
        } else {
          valid = j < p.num_rows;
          if (kKeyScale) {
            kscale = ks_next;
            const int jn = j + EG * 128;
            if (i + EG < it.ntiles && jn < p.num_rows) ks_next = __ldg(p.k_scale + jn);
          }
        }
        bool okt = (lane == 0) ? mbar_wait(tfull0 + 8 * a, (uint32_t)(T >> NBL) & 1u, limit, abort_flag) : true;
        okt = __shfl_sync(0xFFFFFFFFu, okt ? 1 : 0, 0) != 0;
        if (!okt) {
          if (lane == 0) {
            raise_error(DSA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          continue;
        }
        __syncwarp();
        tc_fence_after();
        float v[NQ];
        head_sums<NQ>(t_lane + (uint32_t)(a * N), wq, v);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float sq = v[q];
          if (kKeyScale) sq = sq * kscale;
          v[q] = canon_zero(sq);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * a);

        if (!kTopk) {
          if (j < p.max_len) {
#pragma unroll
            for (int q = 0; q < NQ; ++q)
              if (q < it.nreal)
                p.logits[(int64_t)(it.t0 + q) * p.ld + j] = (valid && j < it.vis[q]) ? v[q] : -INFINITY;
          }
        } else {
          uint64_t key[NQ];
          bool take[NQ];
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            key[q] = rank_key(v[q], (uint32_t)j);
            take[q] = valid && j < it.vis[q] && is_candidate(v[q]) && key[q] >= es->thr[q];
          }
          engine_append_multi<NQ>(ebuf, (size_t)cap, es->cnt, key, take, (uint32_t)cap, 10u);
        }
      }
      T0 += it.ntiles;

      if (!kTopk) {
        // keys of this chunk past the last processed tile are masked for every row
        const int f0 = it.ks + it.ntiles * 128;
        const int f1 = min(it.ks + it.chunk, p.max_len);
        for (int q = 0; q < it.nreal; ++q)
          for (int jj = f0 + et; jj < f1; jj += NT) p.logits[(int64_t)(it.t0 + q) * p.ld + jj] = -INFINITY;
      } else if (!it.split) {
        // the whole group in one item: each row's top k by value bins (the whole epilogue,
        // one row after another; one warp per row sorting in registers took ~94 K cycles per
        // four-row item); a row whose values crowd into one bin, or every row when the plan
        // left no room for the gather buffer, is cut back to SN candidates (histogram, then
        // the exact select) and sorted by the bitonic network
        const int P = p.pow2;
        const int SN = P <= 128 ? 256 : (P <= 512 ? 2 * P : P);   // keys sorted per row (<= cap)
        group_sync<NT>();
#pragma unroll 1
        for (int q = 0; q < NQ; ++q) {
          uint64_t* buf = ebuf + (size_t)q * cap;
          const bool real = q < it.nreal;
          const int64_t t = it.t0 + q;
          int32_t* oi = real ? p.out_idx + t * p.topk : nullptr;
          float* ov = (real && p.out_val) ? p.out_val + t * p.topk : nullptr;
          int m = 0;
          bool done = false;
          if (p.binned)
            done = engine_topk_binned<NT>(buf, (int)min(es->cnt[q], (uint32_t)cap), p.topk, tbuf, kItemMaxBin,
                                          tstart, es->bins, es->esc.hist, es->esc.pick, et, oi, ov, &m);
          if (!done) {
            uint32_t cn = min(es->cnt[q], (uint32_t)cap);
            if (cn > (uint32_t)SN) {
              engine_cut_approx<NT, MAXPER>(buf, &es->cnt[q], (int)cn, p.topk, (uint32_t)SN, es->bins, &es->esc, et);
              cn = min(es->cnt[q], (uint32_t)cap);
            }
            if (cn > (uint32_t)SN) {
              const uint64_t thr = engine_select<NT>(buf, (int)cn, p.topk, &es->esc, et);
              engine_compact<NT, MAXPER>(buf, &es->cnt[q], (int)cn, thr, &es->esc, et);
            }
            group_sync<NT>();
            for (int e = min((int)es->cnt[q], SN) + et; e < SN; e += NT) buf[e] = 0ull;   // rank below all
            group_sync<NT>();
            engine_sort<NT>(buf, cap, 1, SN, et);
            if (real)
              for (int r = et; r < p.topk; r += NT) {
                const uint64_t key = buf[r];
                oi[r] = key ? index_of_key(key) : -1;
                if (ov) ov[r] = key ? value_of_key(key) : -INFINITY;
              }
            m = p.topk;
          }
          if (real)
            for (int r = m + et; r < p.topk; r += NT) {   // fewer than k candidates
              oi[r] = -1;
              if (ov) ov[r] = -INFINITY;
            }
        }
      } else {
        // a piece of a split group: its candidates as they stand (unsorted, at least
        // its top-k) with their count and the piece's threshold, in the slice's list
        // slot; the merge kernel ranks the group's lists
        group_sync<NT>();
        for (int q = 0; q < it.nreal; ++q) {
          const int cn = min((int)es->cnt[q], cap);
          const size_t l = (size_t)it.slot * NQ + q;
          const uint64_t* buf = ebuf + (size_t)q * cap;
          for (int s = et; s < cn; s += NT) p.partial[l * cap + s] = buf[s];
          if (et == 0) {
            p.partial_meta[2 * l] = (uint64_t)cn;
            p.partial_meta[2 * l + 1] = es->thr[q];
          }
        }
      }
      // item slot and its weights free for the producer
      group_sync<NT>();
      if (lane == 0) mbar_arrive(iempty0 + 8 * slot);
    }
    // this warp's TMEM reads are complete
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmemfree);
  }
  else if constexpr (kF4K) {
    // ============================ converters ============================
    // Four warps put each FP4 stage into the block-scaled MMA's operand form.  Thread ct
    // copies key row ct's 64 nibble bytes to a 128-byte row of the padded E2M1 layout
    // (16 codes = 8 packed bytes, the even code in the low nibble as in the cache, then
    // 8 unused bytes) with the 128-byte swizzle (16-byte
    // piece c of row r at r * 128 + ((c ^ (r & 7)) << 4)); each warp writes the tile's
    // E8M0 bytes into its own lane quarter of the tile's scale cells: lane l, column j holds
    // the four scale bytes of key row l + 32 j (the same in every quarter).  A scale byte
    // 0xFF means scale 0 in this cache format but NaN to the tensor cores: its 32 codes are
    // zeroed and the byte becomes 127.  A failed wait skips that step's work; the group
    // stops together at item boundaries.
    constexpr int CBAR = 2;
    const int ct = threadIdx.x - (64 + 128 * EG);
    const uint32_t tq = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16);   // this warp's lane quarter
    tmem_st4(tq + SFB_COL, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);   // the queries: scale 1
    tmem_st4(tq + SFB_COL + 4u, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_st_wait();
    tc_fence_before();
    int T = 0;
    for (int n = 0;; ++n) {
      const int slot = n & 1;
      bool ok = (lane == 0) ? mbar_wait(ifull0 + 8 * slot, (uint32_t)(n >> 1) & 1u, limit, abort_flag) : true;
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok && lane == 0) {
        raise_error(DSA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      group_sync<128>(CBAR);
      if (ct == 0) es->cstop = (*abort_flag != 0) || !es->info[slot].valid;
      group_sync<128>(CBAR);
      if (es->cstop) break;
      const int ntiles = es->info[slot].ntiles;
      for (int i = 0; i < ntiles; ++i, ++T) {
        const int s4 = T % S, c = T % CR;
        bool okt = (lane == 0) ? (mbar_wait(full0 + 8 * s4, (uint32_t)(T / S) & 1u, limit, abort_flag) &&
                                  mbar_wait(cfree0 + 8 * c, ((uint32_t)(T / CR) & 1u) ^ 1u, limit, abort_flag))
                               : true;
        okt = __shfl_sync(0xFFFFFFFFu, okt ? 1 : 0, 0) != 0;
        if (!okt) {
          if (lane == 0) {
            raise_error(DSA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          continue;
        }
        __syncwarp();
        tc_fence_after();                           // the MMAs that read this tile's cells are done
        const uint8_t* f4 = f4_s + (size_t)s4 * F4_BYTES;
        const uint32_t* sc = reinterpret_cast<const uint32_t*>(f4 + 8192);
        const uint32_t sw = sc[ct];
        // Step i handles group g = i ^ m with m = x * ((ct >> 1) & 3) in GF(4) (0, 2, 3, 1):
        // over the 8 threads of a 16-byte access phase, both the row reads (unit 4 (ct & 1)
        // + g of 8) and the swizzled stores (unit (2 g + h) ^ (ct & 7)) then fall in 8
        // different bank groups; the same g for every thread made the reads 4-way conflicts.
        const uint32_t m = (0x1320u >> (4 * ((ct >> 1) & 3))) & 3u;
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4*>(f4 + ct * 64 + (((uint32_t)i ^ m) << 4));
        uint8_t* dst = k_s + (size_t)c * KT_BYTES + ct * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) {               // group g: codes 32 g .. 32 g + 31, pieces 2 g, 2 g + 1
          const uint32_t g = (uint32_t)i ^ m;
          const uint4 x = ((sw >> (8 * g)) & 0xFFu) == 0xFFu ? make_uint4(0u, 0u, 0u, 0u) : v[i];
          *reinterpret_cast<uint4*>(dst + (((2 * g) ^ (ct & 7)) << 4)) = make_uint4(x.x, x.y, 0u, 0u);
          *reinterpret_cast<uint4*>(dst + (((2 * g + 1) ^ (ct & 7)) << 4)) = make_uint4(x.z, x.w, 0u, 0u);
        }
        tmem_st4(tq + SFA_COL + 4u * (uint32_t)c, e8m0_ff_to_one(sc[lane]), e8m0_ff_to_one(sc[lane + 32]),
                 e8m0_ff_to_one(sc[lane + 64]), e8m0_ff_to_one(sc[lane + 96]));
        tmem_st_wait();
        tc_fence_before();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // codes visible to the MMAs
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(cfull0 + 8 * c);
          mbar_arrive(empty0 + 8 * s4);
        }
      }
      group_sync<128>(CBAR);
      if (lane == 0) mbar_arrive(iempty0 + 8 * slot);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(tmemfree);           // no scale cell is written after this
  }
  // No CTA-wide barrier here: the warps leave as their roles end (warp 1 last frees
  // TMEM); shared memory stays valid until every thread of the CTA has exited.
}

// =====================================================================================
// Launch of one instantiation
// =====================================================================================

template <bool kFP8, int NQ, bool kTopk, int EG, bool kF4K = false>
static cudaError_t launch_one(const CUtensorMap& mq, const CUtensorMap& mk, const IndexerParams& prm,
                              const IndexerPlan& pl, int grid, cudaStream_t st) {
  auto kern = indexer_kernel<kFP8, NQ, kTopk, EG, kF4K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(64 + 128 * EG + (kF4K ? 128 : 0));
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kTopk ? 1 : 0;   // top-k mode follows its plan kernel and may overlap it
  e = cudaLaunchKernelEx(&cfg, kern, mq, mk, prm);
  note_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool kFP8, bool kTopk>
static cudaError_t dispatch_nq(const CUtensorMap& mq, const CUtensorMap& mk, const IndexerParams& prm,
                               const IndexerPlan& pl, int grid, cudaStream_t st) {
  if constexpr (kFP8) {
    if (pl.f4k) return pl.nq == 1 ? launch_one<true, 1, kTopk, 2, true>(mq, mk, prm, pl, grid, st)
                                  : launch_one<true, 2, kTopk, 2, true>(mq, mk, prm, pl, grid, st);
  }
  switch (pl.nq * 2 + pl.eg) {
    case 3: return launch_one<kFP8, 1, kTopk, 1>(mq, mk, prm, pl, grid, st);
    case 5: return launch_one<kFP8, 2, kTopk, 1>(mq, mk, prm, pl, grid, st);
    case 6: return launch_one<kFP8, 2, kTopk, 2>(mq, mk, prm, pl, grid, st);
    default: return launch_one<kFP8, 4, kTopk, 2>(mq, mk, prm, pl, grid, st);
  }
}

// One (dtype, mode) pair of the kernel, instantiated in its own translation unit with
// that unit's error word and wait limit.
#define DSA_INDEXER_VARIANT(NAME, FP8, TOPK)                                                          \
  cudaError_t launch_indexer_##NAME(const CUtensorMap& mq, const CUtensorMap& mk, const IndexerParams& prm, \
                                    const IndexerPlan& pl, int grid, cudaStream_t st) {                  \
    return dispatch_nq<FP8, TOPK>(mq, mk, prm, pl, grid, st);                                           \
  }                                                                                                     \
  DSA_DEFINE_TU_ERROR_ACCESSORS(indexer_##NAME)

cudaError_t launch_indexer_bf16_topk(const CUtensorMap&, const CUtensorMap&, const IndexerParams&, const IndexerPlan&,
                                     int, cudaStream_t);
cudaError_t launch_indexer_bf16_logits(const CUtensorMap&, const CUtensorMap&, const IndexerParams&,
                                       const IndexerPlan&, int, cudaStream_t);
cudaError_t launch_indexer_fp8_topk(const CUtensorMap&, const CUtensorMap&, const IndexerParams&, const IndexerPlan&,
                                    int, cudaStream_t);
cudaError_t launch_indexer_fp8_logits(const CUtensorMap&, const CUtensorMap&, const IndexerParams&, const IndexerPlan&,
                                      int, cudaStream_t);

}  // namespace dsa
