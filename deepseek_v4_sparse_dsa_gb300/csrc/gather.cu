// mxfp4 paged gather (xkernels issue #28 "DeepSeek-V4 serving support -- tracking",
// comment 2 "What it does"): selected positions are read through the block table from a
// paged cache of E2M1 nibbles (low nibble = even element) with one E8M0 scale per 32
// elements (2^(b-127), 0xFF -> 0), dequantised to bf16; padded slots give zero rows.
//
// HBM-bound: 68 bytes read and 256 bytes written per live row.  A warp owns 32 rows per
// step.  Each lane resolves one row's source (sel_pos -> block table -> cache row); the
// warp then moves the rows two at a time, 16 lanes per row: a lane loads 4 nibble bytes
// (8 elements) and their scale byte and writes 16 bytes, so every store instruction
// writes two whole 256-byte rows.  The next step's positions and block-table entries
// are fetched while the current rows are in flight.
#include "common.cuh"
#include "launch.h"

namespace dsa {

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

struct GatherArgs {
  const uint8_t* fp4;
  const uint8_t* scale;
  int64_t num_blocks;
  int bs;
  const int32_t* table;
  int64_t bt_stride;
  const int32_t* sel;
  int64_t rows_per_seq;     // next_n * topk
  int64_t rows;
  uint16_t* out;
};

// Cache row of output row r with selected position pos (-1: zero row).
__device__ __forceinline__ int64_t gather_source(const GatherArgs& g, int64_t r, int32_t pos) {
  if (r >= g.rows || pos < 0) return -1;
  const int64_t b = r / g.rows_per_seq;
  const int32_t col = pos / g.bs;
  if (col < g.bt_stride) {
    const int32_t blk = __ldg(g.table + b * g.bt_stride + col);
    if (blk >= 0 && blk < g.num_blocks) return (int64_t)blk * g.bs + pos % g.bs;
  }
  raise_error(DSA_DEVERR_INDEX);
  return -1;
}

__global__ void __launch_bounds__(256) mxfp4_gather_kernel(const GatherArgs g) {
  grid_dependency_wait();              // positions may come from the kernel just before
  const uint32_t lane = threadIdx.x & 31u;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t step = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int sub = (int)(lane >> 4);    // row within a pair
  const int part = (int)(lane & 15u);  // elements 8 * part .. 8 * part + 7
  int64_t r0 = warp * 32;
  int64_t src_next = -1;
  if (r0 < g.rows) {
    const int64_t r = r0 + lane;
    src_next = gather_source(g, r, r < g.rows ? __ldg(g.sel + r) : -1);
  }
  for (; r0 < g.rows; r0 += step * 32) {
    const int64_t src = src_next;
    const int64_t r1 = r0 + step * 32 + lane;
    const int32_t pos_next = r1 < g.rows ? __ldg(g.sel + r1) : -1;   // in flight meanwhile
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t w[8], sb[8];
      int64_t srow[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        srow[k] = __shfl_sync(0xFFFFFFFFu, src, h * 16 + 2 * k + sub);
        w[k] = 0u;
        sb[k] = 255u;
        if (srow[k] >= 0) {
          w[k] = __ldg(reinterpret_cast<const uint32_t*>(g.fp4 + srow[k] * 64) + part);
          sb[k] = __ldg(g.scale + srow[k] * 4 + (part >> 2));
        }
      }
      if (h == 0) src_next = gather_source(g, r1, pos_next);
      // the lane's scale bytes decide, once, between the fast decode and the exact one
      bool exact = false;
#pragma unroll
      for (int k = 0; k < 8; ++k) exact |= e8m0_off_table(sb[k]);
      auto emit = [&](auto decode) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int64_t row = r0 + h * 16 + 2 * k + sub;
          if (row >= g.rows) continue;
          const uint4 v = srow[k] >= 0 ? decode(w[k], sb[k]) : make_uint4(0u, 0u, 0u, 0u);
          st_stream(reinterpret_cast<uint4*>(g.out + row * 128) + part, v);
        }
      };
      if (!exact)
        emit([](uint32_t x, uint32_t b) { return decode8_perm(x, e2m1_bytes(b)); });
      else
        emit([](uint32_t x, uint32_t b) { return decode8_exact(x, b); });
    }
  }
}

cudaError_t launch_mxfp4_gather(const uint8_t* fp4, const uint8_t* scale, int64_t num_blocks, int bs,
                                const int32_t* table, int64_t bt_stride, const int32_t* sel, int next_n,
                                int topk, int64_t rows, uint16_t* out, int num_sms, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  GatherArgs g{fp4, scale, num_blocks, bs, table, bt_stride, sel, (int64_t)next_n * topk, rows, out};
  const int64_t warps_needed = (rows + 31) / 32;
  const int64_t blocks_needed = (warps_needed + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 4;   // resident blocks of 256 threads per SM
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(blocks_needed < cap ? blocks_needed : cap));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, mxfp4_gather_kernel, g);
  note_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

DSA_DEFINE_TU_ERROR_ACCESSORS(gather)

}  // namespace dsa
