// Internal host-side interface between the C ABI (api.cu) and the kernel translation
// units.  Not installed; callers use include/dsa.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

void note_launch();      // counts one kernel launch (dsa_launch_count)
int device_sm_count();   // SMs of the current device (cached per device)

// ------------------------------------------------------------------ indexer (indexer.cu)
struct IndexerPlan {
  int nq;            // query rows per work item (1, 2 or 4)
  int eg;            // epilogue warp groups of 128 threads (1 or 2)
  int stages;        // key-tile pipeline depth
  int nbuf_log2;     // log2 of the TMEM accumulator buffers
  int ctas_per_sm;   // resident CTAs per SM the shared memory allows (1 or 2)
  int chunk;         // logits mode: keys per work item (multiple of 128)
  int nchunks;       // logits mode: ceil(max_context_len / chunk)
  int ngroups;       // ceil(next_n / nq)
  int slices;        // top-k mode: CTAs, one slice of the plan's line each
  int cost;          // top-k mode: fixed cost of one work item, in key tiles
  int cap;           // candidate-buffer capacity per query row (top-k mode)
  int pow2;          // next power of two >= topk
  int check_every;   // top-k mode: tiles between the epilogue's buffer checks (1 or 2)
  bool binned;       // top-k mode: whole groups ranked by value bins (gather buffer in shared
                     // memory; only where it leaves the plan's depth and occupancy unchanged)
  size_t smem;       // dynamic shared memory per CTA
  int64_t items;     // logits mode: work items; top-k mode: query groups
  size_t ws_bytes;   // workspace bytes (top-k mode)
  size_t prefix_off, ufirst_off, split_off, order_off, partial_off, meta_off;   // byte offsets in ws
  bool f4k;          // E4M3 queries, keys from the paged mxfp4 cache (block-scaled MMA)
  int conv_slots;    // FP4-key mode: padded E2M1 key tiles in flight
  bool ok;           // false: shape does not fit this build
};

// topk == 0 plans the logits-only kernel.
// wide = false: no wider candidate buffers (the allocation-free entry, whose scratch is
// bounded, plans without them; results are the same, exact top-k either way).
IndexerPlan plan_indexer(dsa_dtype dt, const dsa_queries& qs, int topk, bool wide = true);

// The fused call and its workspace size with the plan's wider buffers allowed or not
// (api.cu; the public entry points use wide = true).
size_t logits_topk_ws_bytes(dsa_dtype dtype, const dsa_queries& qs, int topk, bool wide);
dsa_status logits_topk_call(const void* q, const float* q_scale, dsa_dtype dtype, const float* weights, int H,
                            int D, const dsa_keys& keys, const dsa_queries& qs, int topk, int32_t* out_idx,
                            float* out_val, void* ws, size_t ws_bytes, void* stream, bool wide);

struct IndexerArgs {
  const void* q;
  const float* q_scale;
  bool fp8;
  const float* weights;
  dsa_keys keys;
  dsa_queries qs;
  // logits mode
  float* logits;
  int64_t ld;
  // top-k mode
  int topk;
  int32_t* out_idx;
  float* out_val;
  void* ws;
};

cudaError_t launch_indexer(const IndexerArgs& a, const IndexerPlan& plan, cudaStream_t stream);

// ------------------------------------------------------------------ top-k (topk.cu)
struct TopkPlan {
  int pow2;          // next power of two >= topk (sorted slots per row)
  size_t smem;       // dynamic shared memory per CTA
  size_t ws_bytes;   // workspace bytes (none needed: 0)
};

TopkPlan plan_topk(const dsa_queries& qs, int topk);

cudaError_t launch_topk(const float* logits, int64_t ld, const dsa_queries& qs, int topk, int32_t* out_idx,
                        float* out_val, void* ws, const TopkPlan& plan, cudaStream_t stream);

// Ranks the partial lists of the query groups the fused kernel split (see the work plan
// in common.cuh): partial = [slices][2][nq][lcap] candidate keys, meta = [slices][2][nq]
// x (count, threshold); plan = header, prefix = group starts on the line, split = the
// split groups (count in the header).  Launched as a programmatic dependent of the
// fused kernel.
cudaError_t launch_merge(const uint64_t* partial, const uint64_t* meta, int lcap, const int32_t* plan,
                         const int32_t* prefix, const int32_t* split, int slices, int nq, const dsa_queries& qs,
                         int topk, int32_t* out_idx, float* out_val, cudaStream_t stream);

// ------------------------------------------------------------------ gather (gather.cu)
cudaError_t launch_mxfp4_gather(const uint8_t* fp4, const uint8_t* scale, int64_t num_blocks, int bs,
                                const int32_t* table, int64_t bt_stride, const int32_t* sel, int next_n,
                                int topk, int64_t rows, uint16_t* out, int num_sms, cudaStream_t stream);

// ------------------------------------------------------------------ producers (producer.cu)
cudaError_t launch_q_rope_quant(const uint16_t* q, const int32_t* positions, const float* cos_sin, int64_t max_pos,
                                int rope_dim, int64_t T, int H, uint8_t* codes, float* scale, int num_sms,
                                cudaStream_t stream);
cudaError_t launch_k_hadamard_mxfp4(const uint16_t* k, const int64_t* slot, int64_t n, uint8_t* fp4, uint8_t* scale,
                                    int64_t num_rows, int num_sms, cudaStream_t stream);

// ------------------------------------------------------------------ sparse attention (sparse_attn.cu)
// q [T, 64, 128] bf16 (16-byte aligned), sel [T, k], the paged mxfp4 cache, sink [64],
// out [T, 64, 128] fp32.  One CTA per query row.
cudaError_t launch_sparse_attn(const uint16_t* q, int64_t T, const int32_t* sel, int k, const uint8_t* fp4,
                               const uint8_t* scale, int64_t num_blocks, int bs, const int32_t* table,
                               int64_t bt_stride, int next_n, const float* sink, float softmax_scale, float* out,
                               int num_sms, cudaStream_t stream);
size_t sparse_attn_smem_bytes(int k);   // dynamic shared memory for a top-k of k slots
int sparse_attn_max_topk();

// ------------------------------------------------------------------ per-TU device words
#define DSA_DECLARE_TU_ERROR_ACCESSORS(name)                                        \
  cudaError_t tu_##name##_read_clear_error(unsigned int* out);                      \
  cudaError_t tu_##name##_set_wait_limit(unsigned long long ns);

#define DSA_DEFINE_TU_ERROR_ACCESSORS(name)                                         \
  cudaError_t tu_##name##_read_clear_error(unsigned int* out) {                     \
    unsigned int zero = 0;                                                          \
    cudaError_t e = cudaMemcpyFromSymbol(out, g_error_word, sizeof(unsigned int));  \
    if (e != cudaSuccess) return e;                                                 \
    return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned int));           \
  }                                                                                 \
  cudaError_t tu_##name##_set_wait_limit(unsigned long long ns) {                   \
    return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns));                    \
  }

DSA_DECLARE_TU_ERROR_ACCESSORS(gather)
DSA_DECLARE_TU_ERROR_ACCESSORS(indexer)
DSA_DECLARE_TU_ERROR_ACCESSORS(indexer_bf16_topk)
DSA_DECLARE_TU_ERROR_ACCESSORS(indexer_bf16_logits)
DSA_DECLARE_TU_ERROR_ACCESSORS(indexer_fp8_topk)
DSA_DECLARE_TU_ERROR_ACCESSORS(indexer_fp8_logits)
DSA_DECLARE_TU_ERROR_ACCESSORS(topk)
DSA_DECLARE_TU_ERROR_ACCESSORS(producer)
DSA_DECLARE_TU_ERROR_ACCESSORS(attn)

// Every translation unit's accessors, for dsa_device_error / dsa_set_wait_limit_ns.
struct TuWords {
  cudaError_t (*read_clear)(unsigned int*);
  cudaError_t (*set_limit)(unsigned long long);
};
#define DSA_TU_WORDS(name) TuWords{tu_##name##_read_clear_error, tu_##name##_set_wait_limit}
inline const TuWords* all_tu_words(int* n) {
  static const TuWords w[] = {DSA_TU_WORDS(gather), DSA_TU_WORDS(indexer), DSA_TU_WORDS(indexer_bf16_topk),
                              DSA_TU_WORDS(indexer_bf16_logits), DSA_TU_WORDS(indexer_fp8_topk),
                              DSA_TU_WORDS(indexer_fp8_logits), DSA_TU_WORDS(topk), DSA_TU_WORDS(producer),
                              DSA_TU_WORDS(attn)};
  *n = (int)(sizeof(w) / sizeof(w[0]));
  return w;
}

}  // namespace dsa
