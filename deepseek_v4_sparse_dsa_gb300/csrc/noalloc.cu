// dsa_indexer_logits_topk_noalloc: the fused indexer score + top-k for callers that must
// not allocate device memory, e.g. a serving process whose device memory is fully
// reserved at start-up and handed out by its own pool, or a latency-critical loop that
// cannot afford cudaMalloc / cudaFree (cudaFree waits for the whole device).
//
// The scratch the fused call needs (its work list and the per-chunk lists of split
// rows) lives in one fixed array in this library's device image instead of a caller
// buffer.  Every GPU that loads the library holds that array until the process exits.
#include <cstdint>
#include <mutex>

#include "launch.h"

namespace dsa {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array on the current device, looked up once per device and kept
// for the life of the process.  (In host code the array's name is only a host-side
// stand-in, never a device address.)  A device reset (cudaDeviceReset) reloads the
// library's device image and may move the array: do not use this entry point across one.
static cudaError_t scratch_on_current_device(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace dsa

extern "C" dsa_status dsa_indexer_logits_topk_noalloc(const void* q, const float* q_scale, dsa_dtype dtype,
                                                      const float* weights, int H, int D, dsa_keys keys,
                                                      dsa_queries qs, int topk, int32_t* out_idx, float* out_val,
                                                      void* stream) {
  // The regular call checks every argument before the workspace, so a bad argument is
  // reported as such whatever the batch size; a batch whose scratch exceeds the array is
  // handed no workspace and gets DSA_ERR_WORKSPACE from that check.  The plan here takes
  // no wider candidate buffers (they would grow the scratch); the result is the same.
  const size_t need = dsa::logits_topk_ws_bytes(dtype, qs, topk, false);
  void* scratch = nullptr;
  if (need > 0 && need <= dsa::kNoAllocScratchBytes) {
    if (dsa::scratch_on_current_device(&scratch) != cudaSuccess) return DSA_ERR_CUDA;
  }
  return dsa::logits_topk_call(q, q_scale, dtype, weights, H, D, keys, qs, topk, out_idx, out_val, scratch,
                               scratch != nullptr ? dsa::kNoAllocScratchBytes : 0, stream, false);
}
