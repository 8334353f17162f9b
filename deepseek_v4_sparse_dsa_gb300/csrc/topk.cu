// Standalone per-row top-k over a logits matrix, and the merge of partial top-k lists.
//
// Rule (README "DeepSeek V4 Flash on a single AMD MI300X", overlay table: deterministic,
// canonical top-k sort): larger value first, then the smaller key index; -0.0 == +0.0;
// -inf / NaN never selected; short rows padded with -1.
//
// Both kernels stream candidates through the shared-memory engine of common.cuh: a
// candidate is appended when its ranking key is >= the current threshold; when the
// buffer could overflow in the next round it is cut back to the top-k by a radix select
// (which also raises the threshold); the survivors are sorted at the end.  Long rows are
// split over several CTAs whose sorted lists are merged by the same engine.
#include "common.cuh"
#include "launch.h"

namespace dsa {

constexpr int kTopkMaxPer = 12;   // capacity <= 256 * 12
constexpr int kRound = 1024;      // candidates per round (4 per thread)

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

__device__ void finish_list(uint64_t* buf, TopkShared* sh, int topk, int P, int tid, int64_t t, int nchunks,
                            int c, int32_t* out_idx, float* out_val, uint64_t* partial) {
  group_sync();
  const uint32_t n = sh->cnt;
  if (n > (uint32_t)topk) {
    const uint64_t thr = engine_select(buf, (int)n, topk, &sh->esc, tid);
    engine_compact<kTopkMaxPer>(buf, &sh->cnt, (int)n, thr, tid);
  }
  const int m = (int)sh->cnt;
  for (int e = m + tid; e < P; e += kEngineThreads) buf[e] = 0ull;
  group_sync();
  engine_sort(buf, P, 1, P, tid);
  for (int s = tid; s < topk; s += kEngineThreads) {
    const uint64_t key = buf[s];
    if (partial) {
      partial[((size_t)t * nchunks + c) * topk + s] = key;
    } else {
      out_idx[t * topk + s] = key ? index_of_key(key) : -1;
      if (out_val) out_val[t * topk + s] = key ? value_of_key(key) : -INFINITY;
    }
  }
}

__global__ void __launch_bounds__(256) topk_rows_kernel(const float* __restrict__ logits, int64_t ld,
                                                        const int32_t* __restrict__ context_lens, int next_n,
                                                        int causal, int max_len, int topk, int chunk,
                                                        int nchunks, int cap, int P, int32_t* out_idx,
                                                        float* out_val, uint64_t* partial) {
  extern __shared__ uint64_t buf[];
  __shared__ TopkShared sh;
  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x / nchunks;
  const int c = blockIdx.x % nchunks;
  const int vis = visible_len(context_lens, (int)t, next_n, causal, max_len, tid == 0 && c == 0);
  const int j0 = c * chunk;
  const int j1 = min(j0 + chunk, vis);
  if (tid == 0) {
    sh.cnt = 0;
    sh.thr = 0;
  }
  const float* row = logits + t * ld;
  float nxt[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int j = j0 + u * 256 + tid;
    nxt[u] = j < j1 ? __ldg(row + j) : -INFINITY;
  }
  for (int base = j0; base < j1; base += kRound) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u] = nxt[u];
      const int j = base + kRound + u * 256 + tid;
      nxt[u] = j < j1 ? __ldg(row + j) : -INFINITY;
    }
    group_sync();
    const uint32_t n = sh.cnt;
    if (n > (uint32_t)(cap - kRound)) {
      const uint64_t thr = engine_select(buf, (int)n, topk, &sh.esc, tid);
      engine_compact<kTopkMaxPer>(buf, &sh.cnt, (int)n, thr, tid);
      if (tid == 0) sh.thr = thr;
      group_sync();
    }
    const uint64_t thr = sh.thr;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = base + u * 256 + tid;
      const uint64_t key = rank_key(v[u], (uint32_t)j);
      engine_append(buf, &sh.cnt, key, j < j1 && is_candidate(v[u]) && key >= thr);
    }
  }
  finish_list(buf, &sh, topk, P, tid, t, nchunks, c, out_idx, out_val, nchunks > 1 ? partial : nullptr);
}

__global__ void __launch_bounds__(256) merge_kernel(const uint64_t* __restrict__ partial, int nchunks, int chunk,
                                                    const int32_t* __restrict__ context_lens, int next_n,
                                                    int causal, int max_len, int topk, int cap, int P,
                                                    int32_t* out_idx, float* out_val) {
  extern __shared__ uint64_t buf[];
  __shared__ TopkShared sh;
  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x;
  const int vis = visible_len(context_lens, (int)t, next_n, causal, max_len, false);
  const int nl = min((vis + chunk - 1) / chunk, nchunks);
  if (tid == 0) {
    sh.cnt = 0;
    sh.thr = 0;
  }
  const uint64_t* src = partial + (size_t)t * nchunks * topk;
  const int64_t total = (int64_t)nl * topk;
  for (int64_t base = 0; base < total; base += kRound) {
    uint64_t v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t e = base + u * 256 + tid;
      v[u] = e < total ? __ldg(src + e) : 0ull;
    }
    group_sync();
    const uint32_t n = sh.cnt;
    if (n > (uint32_t)(cap - kRound)) {
      const uint64_t thr = engine_select(buf, (int)n, topk, &sh.esc, tid);
      engine_compact<kTopkMaxPer>(buf, &sh.cnt, (int)n, thr, tid);
      if (tid == 0) sh.thr = thr;
      group_sync();
    }
    const uint64_t thr = sh.thr;
#pragma unroll
    for (int u = 0; u < 4; ++u) engine_append(buf, &sh.cnt, v[u], v[u] != 0ull && v[u] >= thr);
  }
  finish_list(buf, &sh, topk, P, tid, t, 1, 0, out_idx, out_val, nullptr);
}

static int topk_cap(int topk) {
  const int p2 = next_pow2(topk);
  const int c0 = p2 > topk + kRound ? p2 : topk + kRound;
  return ((c0 + 255) / 256) * 256;
}

TopkPlan plan_topk(const dsa_queries& qs, int topk) {
  TopkPlan pl{};
  pl.pow2 = next_pow2(topk);
  pl.cap = topk_cap(topk);
  pl.smem = (size_t)pl.cap * 8;
  const int64_t T = (int64_t)qs.B * qs.next_n;
  const int64_t full = qs.max_context_len > 0 ? qs.max_context_len : 1;
  int64_t chunk = full;
  if (T < 1216) {
    int64_t want = (full * T + 1215) / 1216;
    want = (want + kRound - 1) / kRound * kRound;
    chunk = want < 8192 ? 8192 : want;
    if (chunk > full) chunk = full;
  }
  pl.chunk = (int)chunk;
  pl.nchunks = (int)((full + chunk - 1) / chunk);
  pl.ws_bytes = pl.nchunks > 1 ? (size_t)T * pl.nchunks * topk * 8 : 0;
  return pl;
}

cudaError_t launch_topk(const float* logits, int64_t ld, const dsa_queries& qs, int topk, int32_t* out_idx,
                        float* out_val, void* ws, const TopkPlan& pl, cudaStream_t stream) {
  const int64_t T = (int64_t)qs.B * qs.next_n;
  if (T <= 0) return cudaSuccess;
  uint64_t* partial = reinterpret_cast<uint64_t*>(ws);
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<(unsigned)(T * pl.nchunks), 256, pl.smem, stream>>>(
      logits, ld, qs.context_lens, qs.next_n, qs.causal, qs.max_context_len, topk, pl.chunk, pl.nchunks, pl.cap,
      pl.pow2, out_idx, out_val, partial);
  note_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess || pl.nchunks == 1) return e;
  return launch_merge(partial, pl.nchunks, pl.chunk, qs, topk, out_idx, out_val, stream);
}

cudaError_t launch_merge(const uint64_t* partial, int nchunks, int chunk, const dsa_queries& qs, int topk,
                         int32_t* out_idx, float* out_val, cudaStream_t stream) {
  const int64_t T = (int64_t)qs.B * qs.next_n;
  if (T <= 0) return cudaSuccess;
  const int cap = topk_cap(topk);
  const size_t smem = (size_t)cap * 8;
  cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  merge_kernel<<<(unsigned)T, 256, smem, stream>>>(partial, nchunks, chunk, qs.context_lens, qs.next_n, qs.causal,
                                                   qs.max_context_len, topk, cap, next_pow2(topk), out_idx,
                                                   out_val);
  note_launch();
  return cudaGetLastError();
}

DSA_DEFINE_TU_ERROR_ACCESSORS(topk)

}  // namespace dsa
