// C ABI of include/dsa.h: argument validation, launch planning and dispatch.
// Every check that can be made on the host is made here, before anything is launched.
#include <cmath>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "launch.h"

namespace dsa {

static std::atomic<unsigned long long> g_launches{0};

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int device_sm_count() {
  static int cache[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

dsa_status check_queries(const dsa_queries& qs) {
  if (qs.B < 0 || qs.max_context_len < 0) return DSA_ERR_INVALID_ARG;
  if (qs.B > 0 && (qs.next_n < 1 || qs.context_lens == nullptr)) return DSA_ERR_INVALID_ARG;
  if ((int64_t)qs.B * qs.next_n > INT32_MAX / 64) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

dsa_status check_keys(const dsa_keys& k, dsa_dtype dt, int B) {
  if (k.data == nullptr || k.num_rows < 1) return DSA_ERR_INVALID_ARG;
  if (!aligned(k.data, 16)) return DSA_ERR_INVALID_ARG;
  if (dt == DSA_E4M3 && k.scale == nullptr) return DSA_ERR_INVALID_ARG;
  if (dt == DSA_E4M3_MXFP4K) {
    if (k.scale_e8m0 == nullptr || !aligned(k.scale_e8m0, 16)) return DSA_ERR_INVALID_ARG;
    if (k.block_table == nullptr && k.num_rows % 4 != 0) return DSA_ERR_UNSUPPORTED;   // 16-byte scale copies
  }
  if (k.num_rows > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (k.block_table != nullptr) {
    const int bs = k.block_size;
    if (bs < 8 || bs % 8 != 0 || !((128 % bs == 0) || (bs % 128 == 0))) return DSA_ERR_UNSUPPORTED;
    if (k.bt_stride < 1 || k.num_rows % bs != 0) return DSA_ERR_INVALID_ARG;
  } else if (B > 1) {
    return DSA_ERR_INVALID_ARG;   // contiguous keys hold one sequence
  }
  return DSA_OK;
}

dsa_status check_indexer_common(const void* q, const float* q_scale, dsa_dtype dtype, const float* weights, int H,
                                int D, const dsa_keys& keys, const dsa_queries& qs) {
  if (dtype != DSA_BF16 && dtype != DSA_E4M3 && dtype != DSA_E4M3_MXFP4K) return DSA_ERR_INVALID_ARG;
  if (H != 64 || D != 128) return DSA_ERR_UNSUPPORTED;
  dsa_status s = check_queries(qs);
  if (s != DSA_OK) return s;
  if (q == nullptr || weights == nullptr || !aligned(q, 16)) return DSA_ERR_INVALID_ARG;
  if (dtype != DSA_BF16 && q_scale == nullptr) return DSA_ERR_INVALID_ARG;
  return check_keys(keys, dtype, qs.B);
}

dsa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

}  // namespace
}  // namespace dsa

using namespace dsa;

dsa_status dsa::logits_topk_call(const void* q, const float* q_scale, dsa_dtype dtype, const float* weights, int H,
                                 int D, const dsa_keys& keys, const dsa_queries& qs, int topk, int32_t* out_idx,
                                 float* out_val, void* ws, size_t ws_bytes, void* stream, bool wide) {
  dsa_status s = check_indexer_common(q, q_scale, dtype, weights, H, D, keys, qs);
  if (s != DSA_OK) return s;
  if (topk < 1 || topk > 2048 || out_idx == nullptr) return DSA_ERR_INVALID_ARG;
  if ((int64_t)qs.B * qs.next_n == 0) return DSA_OK;
  const IndexerPlan pl = plan_indexer(dtype, qs, topk, wide);
  if (!pl.ok) return DSA_ERR_UNSUPPORTED;
  if (pl.ws_bytes > 0 && (ws == nullptr || ws_bytes < pl.ws_bytes || !aligned(ws, 8))) return DSA_ERR_WORKSPACE;
  IndexerArgs a{};
  a.q = q;
  a.q_scale = q_scale;
  a.fp8 = dtype != DSA_BF16;
  a.weights = weights;
  a.keys = keys;
  a.qs = qs;
  a.topk = topk;
  a.out_idx = out_idx;
  a.out_val = out_val;
  a.ws = ws;
  return cuda_status(launch_indexer(a, pl, static_cast<cudaStream_t>(stream)));
}

size_t dsa::logits_topk_ws_bytes(dsa_dtype dtype, const dsa_queries& qs, int topk, bool wide) {
  if (check_queries(qs) != DSA_OK || topk < 1 || topk > 2048) return 0;
  const IndexerPlan pl = plan_indexer(dtype, qs, topk, wide);
  return pl.ok ? pl.ws_bytes : 0;
}

extern "C" {

dsa_status dsa_indexer_logits(const void* q, const float* q_scale, dsa_dtype dtype, const float* weights, int H,
                              int D, dsa_keys keys, dsa_queries qs, float* logits, int64_t ld_logits,
                              void* stream) {
  dsa_status s = check_indexer_common(q, q_scale, dtype, weights, H, D, keys, qs);
  if (s != DSA_OK) return s;
  if (logits == nullptr || ld_logits < qs.max_context_len) return DSA_ERR_INVALID_ARG;
  if ((int64_t)qs.B * qs.next_n == 0 || qs.max_context_len == 0) return DSA_OK;
  const IndexerPlan pl = plan_indexer(dtype, qs, 0);
  if (!pl.ok) return DSA_ERR_UNSUPPORTED;
  IndexerArgs a{};
  a.q = q;
  a.q_scale = q_scale;
  a.fp8 = dtype != DSA_BF16;
  a.weights = weights;
  a.keys = keys;
  a.qs = qs;
  a.logits = logits;
  a.ld = ld_logits;
  a.topk = 0;
  return cuda_status(launch_indexer(a, pl, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_indexer_topk(const float* logits, int64_t ld_logits, dsa_queries qs, int topk, int32_t* out_idx,
                            float* out_val, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = check_queries(qs);
  if (s != DSA_OK) return s;
  if (topk < 1 || topk > 2048) return DSA_ERR_INVALID_ARG;
  if (out_idx == nullptr || ld_logits < qs.max_context_len) return DSA_ERR_INVALID_ARG;
  if (logits == nullptr && qs.max_context_len > 0) return DSA_ERR_INVALID_ARG;
  if ((int64_t)qs.B * qs.next_n == 0) return DSA_OK;
  const TopkPlan pl = plan_topk(qs, topk);
  if (pl.ws_bytes > 0 && (ws == nullptr || ws_bytes < pl.ws_bytes || !aligned(ws, 8))) return DSA_ERR_WORKSPACE;
  return cuda_status(launch_topk(logits, ld_logits, qs, topk, out_idx, out_val, ws, pl,
                                 static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_indexer_logits_topk(const void* q, const float* q_scale, dsa_dtype dtype, const float* weights,
                                   int H, int D, dsa_keys keys, dsa_queries qs, int topk, int32_t* out_idx,
                                   float* out_val, void* ws, size_t ws_bytes, void* stream) {
  return logits_topk_call(q, q_scale, dtype, weights, H, D, keys, qs, topk, out_idx, out_val, ws, ws_bytes, stream,
                          true);
}

dsa_status mxfp4_paged_gather(const uint8_t* kv_fp4, const uint8_t* kv_scale, int64_t num_blocks, int block_size,
                              int D, const int32_t* block_table, int64_t bt_stride, const int32_t* sel_pos, int B,
                              int next_n, int topk, uint16_t* out, void* stream) {
  if (D != 128) return DSA_ERR_UNSUPPORTED;
  if (B < 0 || topk < 0 || num_blocks < 0 || block_size < 1) return DSA_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)B * (B > 0 ? next_n : 0) * topk;
  if (rows == 0) return DSA_OK;
  if (next_n < 1 || bt_stride < 1) return DSA_ERR_INVALID_ARG;
  if (kv_fp4 == nullptr || kv_scale == nullptr || block_table == nullptr || sel_pos == nullptr || out == nullptr)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(kv_fp4, 8) || !aligned(out, 16)) return DSA_ERR_INVALID_ARG;
  return cuda_status(launch_mxfp4_gather(kv_fp4, kv_scale, num_blocks, block_size, block_table, bt_stride, sel_pos,
                                         next_n, topk, rows, out, device_sm_count(),
                                         static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_indexer_q_rope_quant(const uint16_t* q, const int32_t* positions, const float* cos_sin,
                                    int64_t max_pos, int rope_dim, int T, int H, int D, uint8_t* q_fp8,
                                    float* q_scale, void* stream) {
  if (D != 128) return DSA_ERR_UNSUPPORTED;
  if (T < 0 || H < 1 || max_pos < 0) return DSA_ERR_INVALID_ARG;
  if (rope_dim < 0 || rope_dim > D || rope_dim % 4 != 0) return DSA_ERR_INVALID_ARG;
  if ((int64_t)T * H == 0) return DSA_OK;
  if (q == nullptr || positions == nullptr || q_fp8 == nullptr || q_scale == nullptr) return DSA_ERR_INVALID_ARG;
  if (rope_dim > 0 && (cos_sin == nullptr || !aligned(cos_sin, 8))) return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(q_fp8, 8) || !aligned(q_scale, 4)) return DSA_ERR_INVALID_ARG;
  return cuda_status(launch_q_rope_quant(q, positions, cos_sin, max_pos, rope_dim, T, H, q_fp8, q_scale,
                                         device_sm_count(), static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_indexer_k_hadamard_mxfp4(const uint16_t* k, const int64_t* slot_mapping, int64_t N, int D,
                                        uint8_t* kv_fp4, uint8_t* kv_scale, int64_t num_rows, void* stream) {
  if (D != 128) return DSA_ERR_UNSUPPORTED;
  if (N < 0 || num_rows < 0) return DSA_ERR_INVALID_ARG;
  if (N == 0) return DSA_OK;
  if (k == nullptr || slot_mapping == nullptr || kv_fp4 == nullptr || kv_scale == nullptr) return DSA_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(kv_fp4, 4) || !aligned(kv_scale, 4)) return DSA_ERR_INVALID_ARG;
  return cuda_status(launch_k_hadamard_mxfp4(k, slot_mapping, N, kv_fp4, kv_scale, num_rows, device_sm_count(),
                                             static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_sparse_attn_mxfp4(const uint16_t* q, int64_t T, int H, int D, const int32_t* sel_pos, int topk,
                                 const uint8_t* kv_fp4, const uint8_t* kv_scale, int64_t num_blocks, int block_size,
                                 const int32_t* block_table, int64_t bt_stride, int next_n, const float* sink,
                                 float softmax_scale, float* out, void* stream) {
  if (H != 64 || D != 128) return DSA_ERR_UNSUPPORTED;
  if (T < 0 || topk < 0 || num_blocks < 0 || block_size < 1 || T > 0x7FFFFFFF) return DSA_ERR_INVALID_ARG;
  if (topk > sparse_attn_max_topk() || num_blocks * (int64_t)block_size > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (next_n < 1 || bt_stride < 1 || !std::isfinite(softmax_scale)) return DSA_ERR_INVALID_ARG;
  if (q == nullptr || kv_fp4 == nullptr || kv_scale == nullptr || block_table == nullptr || sink == nullptr ||
      out == nullptr || (topk > 0 && sel_pos == nullptr))
    return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_fp4, 16) || !aligned(kv_scale, 4) || !aligned(sink, 4) || !aligned(out, 4))
    return DSA_ERR_INVALID_ARG;
  return cuda_status(launch_sparse_attn(q, T, sel_pos, topk, kv_fp4, kv_scale, num_blocks, block_size, block_table,
                                        bt_stride, next_n, sink, softmax_scale, out, device_sm_count(),
                                        static_cast<cudaStream_t>(stream)));
}

size_t dsa_workspace_bytes(dsa_op op, dsa_dtype dtype, dsa_queries qs, int topk) {
  if (check_queries(qs) != DSA_OK || topk < 1 || topk > 2048) return 0;
  if (op == DSA_OP_TOPK) return plan_topk(qs, topk).ws_bytes;
  if (op == DSA_OP_LOGITS_TOPK) return logits_topk_ws_bytes(dtype, qs, topk, true);
  return 0;
}

const char* dsa_status_string(dsa_status status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case DSA_ERR_CUDA: return "CUDA runtime or launch error";
    case DSA_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

int dsa_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
  unsigned int total = 0;
  int n = 0;
  const TuWords* tus = all_tu_words(&n);
  for (int i = 0; i < n; ++i) {
    unsigned int w = 0;
    if (tus[i].read_clear(&w) != cudaSuccess) return -1;
    total |= w;
  }
  return (int)total;
}

uint64_t dsa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

dsa_status dsa_set_wait_limit_ns(uint64_t ns) {
  const unsigned long long v = ns;
  int n = 0;
  const TuWords* tus = all_tu_words(&n);
  for (int i = 0; i < n; ++i)
    if (tus[i].set_limit(v) != cudaSuccess) return DSA_ERR_CUDA;
  return DSA_OK;
}

}  // extern "C"
