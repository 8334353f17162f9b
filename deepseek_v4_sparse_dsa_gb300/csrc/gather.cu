// mxfp4 paged gather (xkernels issue #28 "DeepSeek-V4 serving support -- tracking",
// comment 2 "What it does"): selected positions are read through the block table from a
// paged cache of E2M1 nibbles (low nibble = even element) with one E8M0 scale per 32
// elements (2^(b-127), 0xFF -> 0), dequantised to bf16; padded slots give zero rows.
//
// HBM-bound: 68 bytes read and 256 bytes written per live row.  A warp owns 32 rows per
// step: each lane resolves one row's source (sel_pos -> block table -> cache row) with
// independent loads, then the warp moves the rows four at a time (8 lanes x 8 nibble
// bytes per row, one 32-byte store per lane), with all eight groups' loads in flight
// before any decode.
#include "common.cuh"
#include "launch.h"

namespace dsa {

// bf16 bit pattern of E2M1 nibble n times 2^(b-127), b != 0xFF, exact except overflow.
// Nonzero magnitudes are (2 + M) * 2^X with (M, X) = (0,-2), (0,-1), (1,-1), (0,0), (1,0),
// (0,1), (1,1) for codes 1..7; the bf16 exponent field is E = X + b + 1 = e + b - 1 for
// code = 2e + m (e >= 1) and b - 1 for code 1.
__device__ __forceinline__ uint32_t e2m1_bf16_general(uint32_t n, int b) {
  const uint32_t s = (n & 8u) << 12;
  const uint32_t c = n & 7u;
  if (c == 0u || b == 255) return s;
  const int e = (int)(c >> 1);
  const uint32_t M = (c > 1u) ? (c & 1u) : 0u;
  const int E = b - 1 + e;
  if (E >= 255) return s | 0x7F80u;                           // beyond bf16 range -> inf
  if (E >= 1) return s | ((uint32_t)E << 7) | (M << 6);        // normal
  return s | ((2u + M) << (E + 5));                            // subnormal (E = 0 or -1)
}

// Fast form for 2 <= b <= 252 (every code lands in the normal range):
// bits = ((b-1) << 7) + (code << 6), minus 64 for code 1; code 0 -> signed zero.
__device__ __forceinline__ uint32_t e2m1_bf16_fast(uint32_t n, uint32_t base) {
  const uint32_t s = (n & 8u) << 12;
  const uint32_t c = n & 7u;
  const uint32_t v = base + (c << 6) - (c == 1u ? 64u : 0u);
  return (c != 0u ? v : 0u) | s;
}

__device__ __forceinline__ void decode16(uint2 w, uint32_t b, uint4& lo, uint4& hi) {
  uint32_t o[8];
  if (b >= 2u && b <= 252u) {
    const uint32_t base = (b - 1u) << 7;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t byte = ((k < 4 ? w.x : w.y) >> (8 * (k & 3))) & 0xFFu;
      o[k] = e2m1_bf16_fast(byte & 0xFu, base) | (e2m1_bf16_fast(byte >> 4, base) << 16);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t byte = ((k < 4 ? w.x : w.y) >> (8 * (k & 3))) & 0xFFu;
      o[k] = e2m1_bf16_general(byte & 0xFu, (int)b) | (e2m1_bf16_general(byte >> 4, (int)b) << 16);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(256) mxfp4_gather_kernel(const uint8_t* __restrict__ fp4,
                                                           const uint8_t* __restrict__ scale,
                                                           int64_t num_blocks, int bs,
                                                           const int32_t* __restrict__ table,
                                                           int64_t bt_stride,
                                                           const int32_t* __restrict__ sel,
                                                           int next_n, int topk, int64_t rows,
                                                           uint16_t* __restrict__ out) {
  const uint32_t lane = threadIdx.x & 31u;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int sub = (int)(lane >> 3);    // row within a group of four
  const int part = (int)(lane & 7u);   // 16 elements: nibble bytes 8*part .. 8*part+7
  for (int64_t r0 = warp * 32; r0 < rows; r0 += nwarps * 32) {
    // 1. each lane resolves one row: -1 = write zeros
    int64_t src = -1;
    const int64_t r = r0 + lane;
    if (r < rows) {
      const int32_t pos = __ldg(sel + r);
      if (pos >= 0) {
        const int64_t b = (r / topk) / next_n;
        const int64_t col = pos / bs;
        bool ok = false;
        if (col < bt_stride) {
          const int32_t blk = __ldg(table + b * bt_stride + col);
          if (blk >= 0 && blk < num_blocks) {
            src = (int64_t)blk * bs + pos % bs;
            ok = true;
          }
        }
        if (!ok) raise_error(DSA_DEVERR_INDEX);
      }
    }
    // 2. eight groups of four rows; issue every load first
    uint2 w[8];
    uint32_t sb[8];
    int64_t srow[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      srow[g] = __shfl_sync(0xFFFFFFFFu, src, g * 4 + sub);
      w[g] = make_uint2(0u, 0u);
      sb[g] = 255u;
      if (srow[g] >= 0) {
        w[g] = __ldg(reinterpret_cast<const uint2*>(fp4 + srow[g] * 64 + part * 8));
        sb[g] = __ldg(scale + srow[g] * 4 + (part >> 1));
      }
    }
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const int64_t row = r0 + g * 4 + sub;
      if (row >= rows) continue;
      uint4 lo, hi;
      if (srow[g] >= 0) {
        decode16(w[g], sb[g], lo, hi);
      } else {
        lo = make_uint4(0u, 0u, 0u, 0u);
        hi = lo;
      }
      uint4* dst = reinterpret_cast<uint4*>(out + row * 128 + part * 16);
      st_stream(dst, lo);
      st_stream(dst + 1, hi);
    }
  }
}

cudaError_t launch_mxfp4_gather(const uint8_t* fp4, const uint8_t* scale, int64_t num_blocks, int bs,
                                const int32_t* table, int64_t bt_stride, const int32_t* sel, int next_n,
                                int topk, int64_t rows, uint16_t* out, int num_sms, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int64_t warps_needed = (rows + 31) / 32;
  const int64_t blocks_needed = (warps_needed + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 8;   // 8 blocks of 256 threads per SM
  const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
  mxfp4_gather_kernel<<<grid, 256, 0, stream>>>(fp4, scale, num_blocks, bs, table, bt_stride, sel, next_n,
                                                topk, rows, out);
  note_launch();
  return cudaGetLastError();
}

DSA_DEFINE_TU_ERROR_ACCESSORS(gather)

}  // namespace dsa
