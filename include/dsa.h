/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek-V4 DSA indexer hot path.
 *
 * The library computes, on one GPU, the three stages of the DeepSeek-V4
 * sparse-attention indexer:
 *
 *   1. the indexer score  logits[t, j] = sum_h w[t, h] * relu(q[t, h, :] . k[j, :])
 *      (xkernels issue #27 "DSA indexer + attention: validate/provide gfx942
 *      forward path", comment 2 "What shipped"; H = index_n_heads = 64,
 *      D = index_head_dim = 128 per the same issue's "Context");
 *   2. a per-query top-k under a fixed tie rule (larger value first, then the
 *      smaller key index), the deterministic "canonical" top-k sort of README
 *      "DeepSeek V4 Flash on a single AMD MI300X" (overlay table);
 *   3. the paged mxfp4 gather of the selected positions to bf16 (xkernels
 *      issue #28 "DeepSeek-V4 serving support -- tracking", comment 2 "What it
 *      does").
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is caller-owned DEVICE memory unless stated
 *   otherwise.  No call allocates or frees memory, synchronises, or keeps a
 *   pointer after it returns.  Calls are asynchronous on `stream` (a
 *   cudaStream_t passed as void*; NULL = the legacy default stream) and run on
 *   the device current to the calling thread.
 * - Query rows: T = B * next_n.  Row t belongs to sequence b = t / next_n and is
 *   query i = t % next_n of it, at absolute position p = L_b - next_n + i, where
 *   L_b = context_lens[b].  With causal != 0 the row sees keys j <= p (and
 *   j < L_b); otherwise every j < L_b.  This is this library's reading of the
 *   "optional per-query causal window" of xkernels issue #27, comment 2.
 * - Host-detectable argument errors return DSA_ERR_INVALID_ARG (or
 *   DSA_ERR_UNSUPPORTED for valid but unimplemented shapes) BEFORE anything is
 *   launched; outputs are then untouched.  A failed launch returns DSA_ERR_CUDA.
 * - Bad indices found on the device (a block id outside [0, num_blocks), a
 *   block-table column outside [0, bt_stride)) never cause an out-of-range
 *   access: the affected key is treated as masked (not selected, logit -inf) or
 *   the gathered row is written as zeros, and a bit is set in the per-device
 *   error word read by dsa_device_error().  A device-side wait that exceeds its
 *   time limit abandons the call's work, sets DSA_DEVERR_TIMEOUT in the same
 *   word and returns without hanging; outputs of that call are then undefined.
 * - v1 supports H = 64 and D = 128 (DSA_ERR_UNSUPPORTED otherwise); they stay
 *   parameters so the ABI does not change when other shapes are added.
 */
#ifndef DSA_GB300_H_
#define DSA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* bad pointer / size / stride / alignment      */
  DSA_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement  */
  DSA_ERR_CUDA = 3,          /* a CUDA runtime or launch error               */
  DSA_ERR_WORKSPACE = 4      /* ws is NULL or smaller than dsa_workspace_bytes */
} dsa_status;

/* Storage of the indexer's inputs.  DSA_BF16: bf16 q and keys.  DSA_E4M3: OCP E4M3 q
 * and keys with fp32 row scales.  DSA_E4M3_MXFP4K: OCP E4M3 q (with q_scale) scored
 * against keys read straight from the paged mxfp4 cache (the fp8-q x fp4-k MQA-logits
 * form that xkernels issue #27 "DSA indexer + attention: validate/provide gfx942
 * forward path", "Status", names; see dsa_keys.scale_e8m0). */
typedef enum { DSA_BF16 = 0, DSA_E4M3 = 1, DSA_E4M3_MXFP4K = 2 } dsa_dtype;

typedef enum { DSA_OP_TOPK = 1, DSA_OP_LOGITS_TOPK = 2 } dsa_op;

/* Bits of the per-device error word (see dsa_device_error). */
#define DSA_DEVERR_INDEX    1u  /* a block id / block-table column was out of range    */
#define DSA_DEVERR_TIMEOUT  2u  /* a bounded device-side wait expired                  */
#define DSA_DEVERR_OVERFLOW 4u  /* an on-chip candidate buffer would have overflowed:
                                   the candidate was dropped (an internal error; bits
                                   8..15 then name the library's internal site)        */

/*
 * Key source of the indexer (the shared MQA key of xkernels issue #27,
 * comment 2).  Keys are rows of D elements, row-major, d fastest; each row
 * starts 16-byte aligned (D * element size is a multiple of 16).
 *  - Paged (block_table != NULL): `data` is a pool of num_rows rows (num_rows =
 *    number of physical blocks * block_size).  Logical key j of sequence b is
 *    pool row block_table[b * bt_stride + j / block_size] * block_size +
 *    j % block_size.  block_size must be a multiple of 8 that divides 128 or is
 *    a multiple of 128; bt_stride >= ceil(L_b / block_size) for every b.
 *  - Contiguous (block_table == NULL): only B == 1; key j is row j, num_rows >= L_0.
 * `scale` is the per-row fp32 scale of E4M3 keys (same row indexing as `data`,
 * non-negative), NULL for bf16.
 * With dtype DSA_E4M3_MXFP4K the keys are rows of the paged mxfp4 cache that
 * mxfp4_paged_gather reads: `data` holds D/2 nibble bytes per row (low nibble = even
 * element, E2M1), `scale_e8m0` D/32 E8M0 bytes per row (2^(b-127), 0xFF -> 0), both
 * 16-byte aligned; `scale` is unused; a contiguous key array needs num_rows % 4 == 0.
 * The key's value is E2M1 * 2^(b-127) exactly; the tensor cores take the codes and
 * scale bytes as stored (block-scaled MMA, one scale per 32 elements).  Scale bytes
 * >= 254 can overflow the fp32 scores and are outside this mode's domain.
 */
typedef struct {
  const void* data;
  const float* scale;
  const int32_t* block_table;
  int64_t bt_stride;
  int32_t block_size;
  int64_t num_rows;
  const uint8_t* scale_e8m0;
} dsa_keys;

/*
 * Query batch layout.  context_lens is DEVICE memory [B] (int32, 0 <= L_b <=
 * max_context_len); max_context_len is a host-side upper bound used to size
 * launches and the logits width.
 */
typedef struct {
  int32_t B;
  int32_t next_n;
  const int32_t* context_lens;
  int32_t max_context_len;
  int32_t causal;
} dsa_queries;

/*
 * dsa_indexer_logits -- indexer score (xkernels issue #27, comment 2 "What
 * shipped"): logits[t * ld_logits + j] = sum_h weights[t*H + h] *
 * relu(qv[t,h,:] . kv[j,:]) for every visible key j, -inf for every other j in
 * [0, max_context_len).  Columns >= max_context_len are not written.
 *  q        [T, H, D] bf16 (dtype DSA_BF16) or E4M3 codes (DSA_E4M3), row-major.
 *  q_scale  [T, H] fp32, non-negative (E4M3 only, else NULL): qv = q * q_scale[t,h].
 *  weights  [T, H] fp32.
 *  keys     see dsa_keys; kv = k (bf16) or k * scale[row] (E4M3).
 *  logits   [T, ld_logits] fp32, ld_logits >= max_context_len.
 * Arithmetic: bf16 or E4M3 products summed in fp32 by the tensor cores, then
 * ReLU, weight and head sum in fp32 in a fixed order (heads 0..63 in four
 * interleaved partial sums), then -0.0 is written as +0.0.  Given the same
 * inputs the scores are bit-identical to those dsa_indexer_logits_topk ranks.
 */
dsa_status dsa_indexer_logits(const void* q, const float* q_scale, dsa_dtype dtype,
                              const float* weights, int H, int D, dsa_keys keys,
                              dsa_queries qs, float* logits, int64_t ld_logits,
                              void* stream);

/*
 * dsa_indexer_topk -- per-row top-k of a logits matrix laid out as
 * dsa_indexer_logits writes it.  Only the visible keys of row t (per `qs`) are
 * candidates; -inf and NaN values are never selected.  out_idx[t * topk + s]
 * (int32) lists the selected key indices in rank order: larger value first,
 * ties to the smaller index, -0.0 equal to +0.0; rows with fewer than topk
 * candidates are padded with -1.  out_val (nullable) receives the matching
 * values (-inf in padded slots).  1 <= topk <= 2048.
 *  ws / ws_bytes: device scratch of at least dsa_workspace_bytes(DSA_OP_TOPK,
 *  DSA_BF16, qs, topk) bytes (may be 0, then ws may be NULL); its contents on
 *  entry do not matter.
 */
dsa_status dsa_indexer_topk(const float* logits, int64_t ld_logits, dsa_queries qs, int topk,
                            int32_t* out_idx, float* out_val, void* ws, size_t ws_bytes,
                            void* stream);

/*
 * dsa_indexer_logits_topk -- dsa_indexer_topk(dsa_indexer_logits(...)) in one
 * pass that never writes the T x max_context_len logits to memory: the scores
 * are ranked on chip as the tensor cores produce them.  Arguments as for the
 * two calls above; the result is bit-identical to running them in sequence.
 * ws: at least dsa_workspace_bytes(DSA_OP_LOGITS_TOPK, dtype, qs, topk) bytes, 8-byte
 * aligned (the work plan, 8 bytes per query group, and two partial top-k lists per
 * CTA of the current device; contents on entry do not matter).
 */
dsa_status dsa_indexer_logits_topk(const void* q, const float* q_scale, dsa_dtype dtype,
                                   const float* weights, int H, int D, dsa_keys keys,
                                   dsa_queries qs, int topk, int32_t* out_idx, float* out_val,
                                   void* ws, size_t ws_bytes, void* stream);

/*
 * mxfp4_paged_gather -- xkernels issue #28, comment 2 "What it does": for every
 * query row t and slot s, pos = sel_pos[t * topk + s];
 *   pos < 0  -> out row is 128 x bf16 +0.0 (a padded slot);
 *   else     -> cache row (blk, off) = (block_table[b * bt_stride + pos / block_size],
 *               pos % block_size) with b = t / next_n, dequantised to bf16:
 *               element e = E2M1(nibble e) * 2^(kv_scale[row][e / 32] - 127),
 *               scale byte 0xFF -> 0 (the sign of the zero follows the nibble),
 *               rounded to nearest-even bf16 (exact except overflow -> inf).
 *  kv_fp4   [num_blocks, block_size, D/2] bytes; byte i of a row holds element
 *           2i in its low nibble and 2i+1 in its high nibble (E2M1: sign bit 3,
 *           two exponent bits, one mantissa bit).
 *  kv_scale [num_blocks, block_size, D/32] E8M0 bytes.
 *  out      [T, topk, D] bf16 bit patterns, row-major.
 * A block id outside [0, num_blocks) or pos / block_size >= bt_stride gives a
 * zero row and sets DSA_DEVERR_INDEX.  D must be 128 (DSA_ERR_UNSUPPORTED
 * otherwise); block_size >= 1.
 */
dsa_status mxfp4_paged_gather(const uint8_t* kv_fp4, const uint8_t* kv_scale, int64_t num_blocks,
                              int block_size, int D, const int32_t* block_table, int64_t bt_stride,
                              const int32_t* sel_pos, int B, int next_n, int topk,
                              uint16_t* out, void* stream);

/*
 * dsa_indexer_q_rope_quant -- the indexer-query producer ahead of the score (vllm PR #1
 * "Sparse-MLA bring-up on MI300X", "Root cause story" item 3: a fused RoPE + FP8
 * quantisation of the indexer query whose bytes the fp8 MQA-logits reader consumes;
 * FP8_MAX = 448 on the OCP path).  For every (token t, head h) row of q:
 *   1. RoPE: for i < rope_dim / 2 the pair (x[2i], x[2i+1]) becomes
 *      (x0 c - x1 s, x0 s + x1 c) with c = cos_sin[p * rope_dim + i],
 *      s = cos_sin[p * rope_dim + rope_dim / 2 + i], p = positions[t]; dims >= rope_dim
 *      pass through (this library's reading: interleaved pairs, a caller-built table);
 *   2. q_scale[t, h] = max_d |y[d]| / 448 (1 for an all-zero row);
 *   3. q_fp8[t, h, d] = E4M3(y[d] / q_scale[t, h]), nearest even, saturating at +-448.
 * All arithmetic in fp32, each product and sum rounded on its own.  The output is the
 * (q, q_scale) pair dsa_indexer_logits* take with dtype DSA_E4M3.
 *  q        [T, H, D] bf16 bit patterns, 16-byte aligned.
 *  positions [T] int32; a position outside [0, max_pos) gives a zero row (codes 0,
 *           scale 0) and sets DSA_DEVERR_INDEX.
 *  cos_sin  [max_pos, rope_dim] fp32 (rope_dim / 2 cosines, then rope_dim / 2 sines per
 *           position), 8-byte aligned; may be NULL when rope_dim == 0.
 *  q_fp8    [T, H, D] E4M3 codes (8-byte aligned); q_scale [T, H] fp32.
 * D must be 128 (DSA_ERR_UNSUPPORTED otherwise); rope_dim a multiple of 4, <= D.
 */
dsa_status dsa_indexer_q_rope_quant(const uint16_t* q, const int32_t* positions, const float* cos_sin,
                                    int64_t max_pos, int rope_dim, int T, int H, int D, uint8_t* q_fp8,
                                    float* q_scale, void* stream);

/*
 * dsa_indexer_k_hadamard_mxfp4 -- the indexer-key compressor's write into the paged FP4
 * cache (ROCm/ATOM issue #707, "CSA": "CSA Indexer Compressor (head_dim=128, Hadamard,
 * FP4)").  For every key n with pool row r = slot_mapping[n] >= 0:
 *   y = H k[n] / sqrt(128), H the Sylvester-ordered Walsh-Hadamard matrix
 *       (H[i][j] = (-1)^popcount(i & j)), in fp32;
 *   per 32-element group g: kv_scale[r, g] = E8M0 byte floor(log2(amax_g)) - 2 + 127
 *       (clamped to >= 0; 0 for an all-zero group), and each element is the nearest E2M1
 *       code of y / 2^(byte - 127) (ties to the even code, saturating at 6; zero results
 *       are +0), packed two per byte of kv_fp4[r], low nibble = even element
 *       (the OCP MX v1.0 conversion, in the layout mxfp4_paged_gather reads).
 *  k            [N, D] bf16 bit patterns, 16-byte aligned.
 *  slot_mapping [N] int64 pool rows (block * block_size + offset); < 0: key skipped;
 *               >= num_rows: skipped and DSA_DEVERR_INDEX set.
 *  kv_fp4       [num_rows, D/2] bytes; kv_scale [num_rows, D/32] bytes (both 4-byte aligned).
 * D must be 128.  The transform is summed by butterflies in fp32: a code can differ
 * from the one of the exactly rounded rotation only where that value lies within a few
 * fp32 ulps of an E2M1 rounding boundary.
 */
dsa_status dsa_indexer_k_hadamard_mxfp4(const uint16_t* k, const int64_t* slot_mapping, int64_t N, int D,
                                        uint8_t* kv_fp4, uint8_t* kv_scale, int64_t num_rows, void* stream);

/*
 * dsa_sparse_attn_mxfp4 -- the sparse-attention consumer of the selection, reading the
 * paged mxfp4 cache directly (ROCm/ATOM issue #707, "CSA": "index-gather + online
 * softmax + attn_sink bias").  This library's reading: for query row t and head h, over
 * the selected positions of row t (sel_pos >= 0), the key and the value are the same
 * dequantised cache row x (the row mxfp4_paged_gather produces); s = softmax_scale *
 * q[t,h,:] . x; the head's sink logit joins the softmax denominator only:
 *   out[t,h,:] = sum_j e^(s_j - m) x_j / (sum_j e^(s_j - m) + e^(sink[h] - m)),
 * m any shift (the result does not depend on it).  A row with no selected position
 * gives zeros.
 *  q        [T, H, D] bf16 bit patterns, 16-byte aligned.  H must be 64 and D 128
 *           (DSA_ERR_UNSUPPORTED otherwise).
 *  sel_pos  [T, topk] int32 positions in row t's sequence b = t / next_n (< 0: padded);
 *           may be NULL when topk == 0.
 *  kv_fp4 [num_blocks, block_size, D/2] (16-byte aligned), kv_scale [num_blocks,
 *           block_size, D/32] (4-byte aligned), block_table [ceil(T / next_n), bt_stride]:
 *           the cache and table exactly as mxfp4_paged_gather reads them.
 *  sink     [H] fp32 logits (-inf: no sink).  softmax_scale finite.
 *  out      [T, H, D] fp32, 4-byte aligned; every element is written.
 * Arithmetic: the scores on the tensor cores from bf16 q and the exactly decoded bf16
 * rows with fp32 accumulation; the softmax in base 2; each weight rounded once to bf16
 * and the same weights summed for the denominator.  So the result is a weighted mean of
 * the selected rows whose weights are off by the bf16 rounding (2^-9 relative) and by
 * the fp32 score error: |out - exact| <= (2^-8 + 2 max_j |ds_j|) max_j |x_j[e]| to first
 * order, ds_j the fp32 error of score j.  Scores must be finite: a row whose scale
 * overflows bf16 (scale bytes 253, 254 with large codes) gives undefined output.
 * A block id outside [0, num_blocks) or a page at or past bt_stride drops that position
 * (as if padded) and sets DSA_DEVERR_INDEX.  topk above 16384 or a cache of 2^31 rows or
 * more (num_blocks * block_size) is DSA_ERR_UNSUPPORTED.  One CTA of 160 threads per
 * query row; two share an SM up to topk 2048.
 */
dsa_status dsa_sparse_attn_mxfp4(const uint16_t* q, int64_t T, int H, int D, const int32_t* sel_pos, int topk,
                                 const uint8_t* kv_fp4, const uint8_t* kv_scale, int64_t num_blocks,
                                 int block_size, const int32_t* block_table, int64_t bt_stride, int next_n,
                                 const float* sink, float softmax_scale, float* out, void* stream);

/*
 * dsa_indexer_logits_topk_noalloc -- dsa_indexer_logits_topk for callers that cannot
 * allocate device memory: a process whose device memory is all reserved at start-up
 * and handed out by its own pool, or a latency-critical loop that cannot afford
 * cudaMalloc / cudaFree (cudaFree waits for the whole device).  (The pages have no
 * counterpart: this is a convenience of this library.)
 * Same arguments and results as dsa_indexer_logits_topk, without ws / ws_bytes: the
 * scratch lives in a fixed 16 MiB array in the library's device image, which every
 * GPU that loads the library holds until the process exits.
 *  - Its plan takes no wider candidate buffers than the batch needs (the regular call
 *    widens them where shared memory allows, which grows its workspace); results are the
 *    same.  A batch whose scratch under that plan exceeds 16 MiB is rejected with
 *    DSA_ERR_WORKSPACE before anything is launched; that scratch is never more than
 *    dsa_workspace_bytes(DSA_OP_LOGITS_TOPK, ...).
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *    and keeps it for the process; make that first call before any stream capture, and do
 *    not use this call across a device reset (cudaDeviceReset may move the array).
 *  - Which batches fit depends on the device's SM count (the plan keeps two partial top-k
 *    lists per SM): on a 152-SM GB300 the tiny, Flash decode, Pro decode MTP and 16K
 *    prefill batches fit; the FP8 chunked prefill (8192 rows, top-1024) does not.
 *  - All calls share the one array; the call itself rewrites every part it reads
 *    (its work plan and partial top-k lists), so stale contents never matter.
 *    Calls whose executions overlap on the GPU (other streams, other threads) race on
 *    the array: serialise them.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
dsa_status dsa_indexer_logits_topk_noalloc(const void* q, const float* q_scale, dsa_dtype dtype,
                                           const float* weights, int H, int D, dsa_keys keys,
                                           dsa_queries qs, int topk, int32_t* out_idx, float* out_val,
                                           void* stream);

/* Workspace bytes the op needs for this batch shape on the current device (host only,
 * no device work; the fused call's plan has one slice per resident CTA, so the size
 * depends on the device's SM count). */
size_t dsa_workspace_bytes(dsa_op op, dsa_dtype dtype, dsa_queries qs, int topk);

/* Static text for a status code. */
const char* dsa_status_string(dsa_status status);

/* Synchronises `stream`, then returns and clears the current device's error
 * word (DSA_DEVERR_* bits; 0 = no device-side error since the last read).
 * Returns -1 if the synchronisation or the read fails. */
int dsa_device_error(void* stream);

/* Number of kernels this library has launched in this process (all threads,
 * all devices); lets a caller count the launches inside a timed region. */
uint64_t dsa_launch_count(void);

/* Sets the limit, in nanoseconds, of every bounded device-side wait launched
 * after this call on the current device (default 2 s; 0 restores the
 * default).  Returns DSA_ERR_CUDA if the device symbol cannot be written. */
dsa_status dsa_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H_ */
