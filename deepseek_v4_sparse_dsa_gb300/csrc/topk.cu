// Standalone per-row top-k over a logits matrix, and the merge of partial top-k lists.
//
// Rule (README "DeepSeek V4 Flash on a single AMD MI300X", overlay table: deterministic,
// canonical top-k sort): larger value first, then the smaller key index; -0.0 == +0.0;
// -inf / NaN never selected; short rows padded with -1.
//
// Both use the top-k engine of common.cuh.  The standalone top-k reads each row straight
// from memory (a few select passes, one collect pass); the merge ranks the per-slice
// candidate lists the fused indexer kernel wrote for the query groups it split.
#include "common.cuh"
#include "launch.h"

namespace dsa {


__device__ __forceinline__ int visible_len(const int32_t* context_lens, int t, int next_n, int causal,
                                           int max_len, bool report) {
  const int b = t / next_n, i = t - b * next_n;
  int L = __ldg(context_lens + b);
  if (L < 0 || L > max_len) {
    if (report) raise_error(DSA_DEVERR_INDEX);
    L = L < 0 ? 0 : max_len;
  }
  return causal ? min(max(L - next_n + i + 1, 0), L) : L;
}

struct TopkShared {
  uint32_t cnt;
  uint64_t thr;
  EngineScratch esc;
};

constexpr int kRowNT = 1024;        // standalone top-k: threads per row

// Ranking key of logits[t, j]: 0 (never selected) past the visible range or for -inf/NaN.
__device__ __forceinline__ uint64_t row_key(const float* __restrict__ row, int j, int vis) {
  if (j >= vis) return 0ull;
  const float v = __ldg(row + j);
  return is_candidate(v) ? rank_key(v, (uint32_t)j) : 0ull;
}

// One CTA per query row.  The row's visible logits are read straight from memory in a
// few passes: a most-significant-digit radix select over the 64-bit ranking keys finds
// the k-th key (passes stop as soon as the chosen bin holds exactly the keys still
// needed), one more pass collects the keys at or above it -- exactly min(k, candidates)
// of them -- into shared memory, where they are sorted and written.
__global__ void __launch_bounds__(kRowNT) topk_rows_kernel(const float* __restrict__ logits, int64_t ld,
                                                           const int32_t* __restrict__ context_lens, int next_n,
                                                           int causal, int max_len, int topk, int P,
                                                           int32_t* out_idx, float* out_val) {
  extern __shared__ uint64_t sel[];     // P slots
  __shared__ EngineScratch esc;
  __shared__ uint32_t cnt;
  constexpr int NT = kRowNT;
  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x;
  const int vis = visible_len(context_lens, (int)t, next_n, causal, max_len, tid == 0);
  const float* row = logits + t * ld;
  // radix select over the keys of this row
  uint64_t prefix = 0, mask = 0;
  uint32_t need = (uint32_t)topk;
  bool all = false;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) esc.hist[i] = 0;
    group_sync<NT>();
    for (int base = 0; base < vis; base += 4 * NT) {
      uint64_t key[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) key[u] = row_key(row, base + u * NT + tid, vis);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        hist_add(esc.hist, key[u] != 0ull && (key[u] & mask) == prefix, (uint32_t)(key[u] >> shift) & 255u);
    }
    group_sync<NT>();
    if (tid < 32) pick_digit(esc.hist, esc.pick, need, tid);
    group_sync<NT>();
    if (shift == 56 && esc.pick[3] <= (uint32_t)topk) {
      all = true;                       // at most k candidates: take every one
      break;
    }
    const uint32_t d = esc.pick[0], above = esc.pick[1], inbin = esc.pick[2];
    if (d > 255u) {                     // counts did not add up (cannot happen): keep every candidate
      if (tid == 0) raise_error(DSA_DEVERR_OVERFLOW | (40u << 8));
      all = true;
      break;
    }
    need -= above;
    prefix |= (uint64_t)d << shift;
    mask |= (uint64_t)0xFF << shift;
    if (inbin == need) break;
  }
  const uint64_t thr = all ? 1ull : prefix;
  if (tid == 0) cnt = 0;
  group_sync<NT>();
  for (int base = 0; base < vis; base += NT) {
    const uint64_t key = row_key(row, base + tid, vis);
    engine_append(sel, &cnt, key, key != 0ull && key >= thr, (uint32_t)P, 41u);
  }
  group_sync<NT>();
  const int m = min((int)cnt, P);
  for (int e = m + tid; e < P; e += NT) sel[e] = 0ull;
  group_sync<NT>();
  engine_sort<NT>(sel, P, 1, P, tid);
  for (int s = tid; s < topk; s += NT) {
    const uint64_t key = sel[s];
    out_idx[t * topk + s] = key ? index_of_key(key) : -1;
    if (out_val) out_val[t * topk + s] = key ? value_of_key(key) : -INFINITY;
  }
}

// Writes every selected key out[0, m) (m <= 4 * NT, distinct unless the lists were stale)
// at its rank, the number of larger keys.  The keys are binned by value image into kCutBins
// linear bins over their range (as in a cut-back); a key's rank is the count in the bins
// above its own plus the larger keys of its own bin, found by scanning that bin: a few
// keys on average, all m at worst (then it costs what counting against every key costs).
// Scratch: tmp (m slots), start and bins (kCutBins words each), red (2 * NT / 32 words).
template <int NT>
__device__ void merge_rank_binned(const uint64_t* out, int m, uint64_t* tmp, uint32_t* start, uint32_t* bins,
                                  uint32_t* red, int tid, int topk, int32_t* row_idx, float* row_val) {
  constexpr int NW = NT / 32, KPT = 4;
  static_assert(kCutBins == NT, "one bin per thread in the scan");
  const int lane = tid & 31, w = tid >> 5;
  uint64_t key[KPT];
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
  for (int u = 0; u < KPT; ++u) {
    const int e = tid + u * NT;
    key[u] = e < m ? out[e] : 0ull;
    if (key[u]) {
      lo = min(lo, (uint32_t)(key[u] >> 32));
      hi = max(hi, (uint32_t)(key[u] >> 32));
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
  }
  if (lane == 0) {
    red[w] = lo;
    red[NW + w] = hi;
  }
  bins[tid] = 0u;
  group_sync<NT>();
  lo = 0xFFFFFFFFu;
  hi = 0u;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    lo = min(lo, red[i]);
    hi = max(hi, red[NW + i]);
  }
  const uint64_t span = hi >= lo ? (uint64_t)(hi - lo) + 1u : 1u;
  const uint32_t mul = (uint32_t)min(((uint64_t)kCutBins << 32) / span, (uint64_t)0xFFFFFFFFu);
  uint32_t bk[KPT];
#pragma unroll
  for (int u = 0; u < KPT; ++u) {
    bk[u] = key[u] ? cut_bin((uint32_t)(key[u] >> 32), lo, mul) : 0u;
    if (key[u]) atomicAdd(&bins[bk[u]], 1u);
  }
  group_sync<NT>();
  // start[b]: the keys in the bins above b (thread tid scans bin kCutBins - 1 - tid)
  const int b = kCutBins - 1 - tid;
  const uint32_t c = bins[b];
  uint32_t incl = c;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  group_sync<NT>();                              // red is rewritten
  if (lane == 31) red[w] = incl;
  group_sync<NT>();
  uint32_t before = 0;
  for (int i = 0; i < w; ++i) before += red[i];
  start[b] = before + incl - c;
  bins[b] = before + incl - c;                   // running slot of the scatter
  group_sync<NT>();
#pragma unroll
  for (int u = 0; u < KPT; ++u)
    if (key[u]) tmp[atomicAdd(&bins[bk[u]], 1u)] = key[u];
  group_sync<NT>();
#pragma unroll
  for (int u = 0; u < KPT; ++u) {
    if (!key[u]) continue;
    const uint32_t s0 = start[bk[u]], s1 = bins[bk[u]];
    uint32_t r = s0;
    for (uint32_t j = s0; j < s1; ++j) r += tmp[j] > key[u] ? 1u : 0u;
    if (r >= (uint32_t)topk) {                  // only if the lists held equal keys (stale lists
      raise_error(DSA_DEVERR_OVERFLOW | (33u << 8));   // after an abandoned call): never write
      continue;                                 // past the row
    }
    row_idx[r] = index_of_key(key[u]);
    if (row_val) row_val[r] = value_of_key(key[u]);
  }
}

constexpr int kMergeNT = 512;       // merge: threads per row
constexpr int kMergeLoads = 8;      // merge: list keys each thread loads per round
constexpr int kMergeKeys = 24576;   // merge: candidates held in shared memory at once (two halves)

// One CTA per (split group, query row): block m handles row m % nq of the (m / nq)-th
// split group of the plan.  The row's lists (one per slice the group's tiles fall in)
// hold each piece's candidates -- a superset of its top-k -- and the piece's threshold
// (its k-th best key at its last cut-back, or 0).  The largest of those thresholds is a
// lower bound of the row's k-th best key: only keys at or above it are loaded.  They
// collect in one half of the shared buffer, which is cut back to the top-k whenever it
// fills; a last radix select leaves exactly the row's top-k, each of which is written at
// its rank (the number of selected keys above it).
__global__ void __launch_bounds__(kMergeNT) merge_kernel(const uint64_t* __restrict__ partial,
                                                         const uint64_t* __restrict__ meta, int lcap,
                                                         const int32_t* plan, const int32_t* prefix,
                                                         const int32_t* split, int nq, int next_n, int topk, int P,
                                                         int32_t* out_idx, float* out_val) {
  extern __shared__ uint64_t mbuf[];            // kMergeKeys candidates + P selected
  __shared__ TopkShared sh;
  __shared__ uint64_t s_floor[kMergeNT / 32];
  __shared__ uint32_t s_off[33], s_li[32];
  __shared__ __align__(16) uint32_t mbins[kCutBins];   // also read as 64-bit words
  constexpr int NT = kMergeNT;
  constexpr int kHalf = kMergeKeys / 2;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  grid_dependency_wait();                       // the fused kernel's lists are complete
  grid_launch_dependents();                     // a gather of the results may set up meanwhile
  const int blk = (int)blockIdx.x;
  const int si = blk / nq, q = blk - si * nq;
  if (si >= __ldcg(plan + 2)) return;
  const int Q = __ldcg(plan), cost = __ldcg(plan + 3);
  const int g = __ldcg(split + si);
  const int ngroups = (next_n + nq - 1) / nq;
  const int b = g / ngroups, gi = g - b * ngroups;
  if (gi * nq + q >= next_n) return;            // padding row of the last group
  const int64_t t = (int64_t)b * next_n + gi * nq + q;
  const int a0 = __ldcg(prefix + g), a1 = __ldcg(prefix + g + 1);
  const int s0 = first_tile_slice(a0, cost, Q);
  const int nl = last_tile_slice(a1, Q) - s0 + 1;
  auto list_of = [&](int l) -> size_t { return (size_t)split_slot(s0 + l, a0, cost, Q) * nq + q; };
  // Collect the keys at or above the running threshold, cutting back when full; lists
  // are taken 32 at a time, their keys as one flat range.  The threshold starts at the
  // largest piece threshold of the lists read so far (each is at most the row's k-th key,
  // so any of them is a floor), read with the lists' counts.
  uint64_t* cur = mbuf;
  uint64_t* alt = mbuf + kHalf;
  for (int c0 = 0; c0 < nl; c0 += 32) {
    const int nc = min(32, nl - c0);
    if (wid == 0) {
      uint32_t cn = 0;
      size_t li = 0;
      uint64_t fl = 0;
      if (lane < nc) {
        li = list_of(c0 + lane);
        cn = (uint32_t)min((uint64_t)lcap, __ldcg(meta + 2 * li));
        fl = __ldcg(meta + 2 * li + 1);
      }
      uint32_t incl = cn;
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      for (int o = 16; o > 0; o >>= 1) fl = max(fl, __shfl_xor_sync(0xFFFFFFFFu, fl, o));
      s_off[lane + 1] = incl;
      s_li[lane] = (uint32_t)li;
      if (lane == 0) {
        s_off[0] = 0;
        if (c0 == 0) sh.cnt = 0;
        sh.thr = c0 == 0 ? fl : max(sh.thr, fl);
      }
    }
    group_sync<NT>();
    const int total = (int)s_off[nc];
    for (int base = 0; base < total; base += kMergeLoads * NT) {
      uint64_t v[kMergeLoads];
#pragma unroll
      for (int u = 0; u < kMergeLoads; ++u) {
        const int e = base + u * NT + tid;
        v[u] = 0ull;
        if (e < total) {
          int l = 0;                            // last list with s_off[l] <= e
#pragma unroll
          for (int step = 16; step > 0; step >>= 1)
            if (l + step < nc && (int)s_off[l + step] <= e) l += step;
          v[u] = __ldcg(partial + (size_t)s_li[l] * lcap + (e - (int)s_off[l]));
        }
      }
      group_sync<NT>();
      // The count runs past kHalf only when appends were dropped (flagged as an overflow):
      // lists left stale by an abandoned call can hold thousands of equal keys, which no
      // cut can thin.  Nothing past the half is ever read.
      const uint32_t n = min(sh.cnt, (uint32_t)kHalf);
      if (n > (uint32_t)(kHalf - kMergeLoads * NT)) {
        uint64_t th = engine_cut_approx<NT, kHalf / NT>(cur, &sh.cnt, (int)n, topk, (uint32_t)(kHalf / 2), mbins,
                                                        &sh.esc, tid);
        if (th == 0ull) {
          th = engine_select<NT>(cur, (int)n, topk, &sh.esc, tid);
          engine_compact_to<NT>(cur, alt, &sh.cnt, (int)n, th, tid, (uint32_t)kHalf);
          uint64_t* tmp = cur;
          cur = alt;
          alt = tmp;
        }
        if (tid == 0 && th > sh.thr) sh.thr = th;
        group_sync<NT>();
      }
      const uint64_t th = sh.thr;
#pragma unroll
      for (int u = 0; u < kMergeLoads; ++u)
        engine_append(cur, &sh.cnt, v[u], v[u] != 0ull && v[u] >= th, (uint32_t)kHalf, 31u);
    }
    group_sync<NT>();                           // s_off / s_li are rewritten next round
  }
  // Then the row's top-k in rank order: by value bins straight from the candidates; when
  //    the values crowd into one bin, a histogram cut, the exact radix select, and the
  //    binned rank of the selected keys
  uint32_t n = min(sh.cnt, (uint32_t)kHalf);
  int32_t* row_idx = out_idx + t * topk;
  float* row_val = out_val ? out_val + t * topk : nullptr;
  int m = 0;
  if (!engine_topk_binned<NT>(cur, (int)n, topk, alt, 2048u, reinterpret_cast<uint32_t*>(alt + 8192), mbins,
                              reinterpret_cast<uint32_t*>(s_floor), sh.esc.pick, tid, row_idx, row_val, &m)) {
    if (n > (uint32_t)topk) {
      engine_cut_approx<NT, kHalf / NT>(cur, &sh.cnt, (int)n, topk, n, mbins, &sh.esc, tid);
      n = min(sh.cnt, (uint32_t)kHalf);
    }
    const uint64_t thr = engine_select<NT>(cur, (int)n, topk, &sh.esc, tid);
    uint64_t* out = mbuf + kMergeKeys;
    if (tid == 0) sh.cnt = 0;
    group_sync<NT>();
    for (int base = 0; base < (int)n; base += NT) {
      const int e = base + tid;
      const uint64_t key = e < (int)n ? cur[e] : 0ull;
      engine_append(out, &sh.cnt, key, key != 0ull && key >= thr, (uint32_t)P, 32u);
    }
    group_sync<NT>();
    m = min((int)sh.cnt, P);
    merge_rank_binned<NT>(out, m, cur, reinterpret_cast<uint32_t*>(alt), mbins, reinterpret_cast<uint32_t*>(s_floor),
                          tid, topk, row_idx, row_val);
  }
  for (int s = m + tid; s < topk; s += NT) {
    out_idx[t * topk + s] = -1;
    if (out_val) out_val[t * topk + s] = -INFINITY;
  }
}

TopkPlan plan_topk(const dsa_queries& qs, int topk) {
  TopkPlan pl{};
  pl.pow2 = next_pow2(topk);
  pl.smem = (size_t)pl.pow2 * 8;
  pl.ws_bytes = 0;
  return pl;
}

cudaError_t launch_topk(const float* logits, int64_t ld, const dsa_queries& qs, int topk, int32_t* out_idx,
                        float* out_val, void* ws, const TopkPlan& pl, cudaStream_t stream) {
  (void)ws;
  const int64_t T = (int64_t)qs.B * qs.next_n;
  if (T <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<(unsigned)T, kRowNT, pl.smem, stream>>>(logits, ld, qs.context_lens, qs.next_n, qs.causal,
                                                            qs.max_context_len, topk, pl.pow2, out_idx, out_val);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge(const uint64_t* partial, const uint64_t* meta, int lcap, const int32_t* plan,
                         const int32_t* prefix, const int32_t* split, int slices, int nq, const dsa_queries& qs,
                         int topk, int32_t* out_idx, float* out_val, cudaStream_t stream) {
  if ((int64_t)qs.B * qs.next_n <= 0 || slices <= 0) return cudaSuccess;
  const int P = next_pow2(topk);
  const size_t smem = (size_t)(kMergeKeys + P + 2) * 8;
  cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(slices * nq));    // at most slices - 1 split groups
  cfg.blockDim = dim3(kMergeNT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, merge_kernel, partial, meta, lcap, plan, prefix, split, nq, (int)qs.next_n, topk, P,
                         out_idx, out_val);
  note_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

DSA_DEFINE_TU_ERROR_ACCESSORS(topk)

}  // namespace dsa
