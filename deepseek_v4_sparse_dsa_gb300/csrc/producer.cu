// Producers around the indexer score (sm_103a): the indexer-query RoPE + per-row FP8
// quantisation ahead of it, and the indexer-key Hadamard rotation + mxfp4 write into
// the paged cache that the score (FP4-key form) and the gather read.
//
// Indexer-Q producer (vllm PR #1 "Sparse-MLA bring-up on MI300X", "Root cause story"
// item 3: a fused RoPE + FP8 quantisation of the indexer query, FP8_MAX = 448 on the OCP
// path).  16 lanes per (token, head) row of 128 dims, 8 dims per lane: the interleaved
// pairs (2i, 2i+1) of the first rope_dim dims turn by the table's cos / sin for the
// token's position, the row's largest magnitude gives scale = amax / 448, and each dim
// becomes E4M3(value / scale) (nearest even, saturating).  Every product and sum is
// rounded on its own (no contraction into FMAs): the codes are integers decided by that
// fp32 arithmetic.
//
// Indexer-key writer (ROCm/ATOM issue #707, "CSA": "CSA Indexer Compressor
// (head_dim=128, Hadamard, FP4)").  16 lanes per key of 128 dims, 8 per lane: a
// 128-point Walsh-Hadamard transform (Sylvester order; three butterfly stages inside a
// lane, four across lanes by shuffles) scaled by 1/sqrt(128), then the OCP MX encoding
// of the gather's layout: per 32-element group (4 lanes) the E8M0 byte is
// max(exponent field of amax - 2, 0) (= floor(log2 amax) - 2 + 127), each element the
// nearest E2M1 code of value / 2^(byte - 127) (ties to the even code, saturating at 6, by
// the hardware conversion; zero results +0), packed two per byte, low nibble = even element.
//
// Both are HBM-bound streams (a few hundred bytes per row): each lane loads 16 bytes per
// row, and a warp issues the loads of 8 rows before using any of them.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace dsa {

// Rows are handled 16 lanes to a row (8 elements, 16 bytes of bf16 per lane), two rows per
// warp instruction, and kProdPairs such pairs per warp step, all loaded before any is used.
constexpr int kProdPairs = 4;
constexpr int kProdRowsPerStep = 2 * kProdPairs;

struct QRopeArgs {
  const uint16_t* q;
  const int32_t* positions;
  const float* cos_sin;
  int64_t max_pos;
  int rope_dim;
  int H;
  int64_t rows;             // T * H
  uint8_t* codes;
  float* scale;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__global__ void __launch_bounds__(256) q_rope_quant_kernel(const QRopeArgs a) {
  const int lane = threadIdx.x & 31, hl = lane & 15, sub = lane >> 4;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int p0 = hl * 4;                         // this lane's pairs p0 .. p0 + 3 (dims 8 hl .. 8 hl + 7)
  const int half = a.rope_dim >> 1;              // rotated pairs: p < half
  for (int64_t r0 = warp * kProdRowsPerStep; r0 < a.rows; r0 += nwarps * kProdRowsPerStep) {
    uint4 raw[kProdPairs];
    float cs[kProdPairs][8];                     // cos of pairs p0 .. p0 + 3, then their sin
    bool ok[kProdPairs];
#pragma unroll
    for (int u = 0; u < kProdPairs; ++u) {
      const int64_t r = r0 + 2 * u + sub;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        cs[u][i] = 1.f;
        cs[u][4 + i] = 0.f;
      }
      ok[u] = false;
      if (r < a.rows) {
        raw[u] = __ldg(reinterpret_cast<const uint4*>(a.q + r * 128) + hl);
        const int64_t pos = __ldg(a.positions + r / a.H);
        ok[u] = pos >= 0 && pos < a.max_pos;
        if (ok[u]) {
          const float* row = a.cos_sin + pos * a.rope_dim;
#pragma unroll
          for (int j = 0; j < 4; j += 2) {       // two pairs per 8-byte load, only inside the table row
            if (p0 + j < half) {
              const float2 c = __ldg(reinterpret_cast<const float2*>(row + p0 + j));
              const float2 sn = __ldg(reinterpret_cast<const float2*>(row + half + p0 + j));
              cs[u][j] = c.x;
              cs[u][j + 1] = c.y;
              cs[u][4 + j] = sn.x;
              cs[u][4 + j + 1] = sn.y;
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kProdPairs; ++u) {
      const int64_t r = r0 + 2 * u + sub;
      const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
      float y[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        y[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        y[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {              // pair p0 + j = dims (2 (p0 + j), 2 (p0 + j) + 1)
        if (p0 + j < half) {
          const float x0 = y[2 * j], x1 = y[2 * j + 1], c = cs[u][j], sn = cs[u][4 + j];
          y[2 * j] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn));
          y[2 * j + 1] = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, c));
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(y[i]));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));   // within the 16 lanes
      const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
      uint32_t packed[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(y[e], sc), __NV_SATFINITE, __NV_E4M3);
        packed[e >> 2] |= (uint32_t)c << (8 * (e & 3));
      }
      if (r < a.rows) {
        if (!ok[u]) {
          packed[0] = packed[1] = 0u;
          if (hl == 0) raise_error(DSA_DEVERR_INDEX);
        }
        reinterpret_cast<uint2*>(a.codes + r * 128)[hl] = make_uint2(packed[0], packed[1]);
        if (hl == 0) a.scale[r] = ok[u] ? sc : 0.f;
      }
    }
  }
}

struct KWriteArgs {
  const uint16_t* k;
  const int64_t* slot;
  int64_t n;
  int64_t num_rows;
  uint8_t* fp4;
  uint8_t* scale;
};

// Nearest E2M1 codes of a pair (ties to the even code, saturating at +-6) by the tensor-core
// conversion instruction: `hi` in the high nibble, `lo` in the low one.
__device__ __forceinline__ uint32_t e2m1x2(float hi, float lo) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Clears the sign of every nibble of `nib` (8 nibbles) whose magnitude is 0: a value that
// rounds to zero is written as +0.
__device__ __forceinline__ uint32_t positive_zeros8(uint32_t nib) {
  const uint32_t mag = nib & 0x77777777u;
  const uint32_t nz = (mag | (mag >> 1) | (mag >> 2)) & 0x11111111u;
  return nib & ((nz << 3) | 0x77777777u);
}

__global__ void __launch_bounds__(256) k_hadamard_mxfp4_kernel(const KWriteArgs a) {
  const int lane = threadIdx.x & 31, hl = lane & 15, sub = lane >> 4;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const float norm = 0.08838834764831845f;       // 1 / sqrt(128), rounded to fp32
  for (int64_t n0 = warp * kProdRowsPerStep; n0 < a.n; n0 += nwarps * kProdRowsPerStep) {
    uint4 raw[kProdPairs];
    int64_t row[kProdPairs];
#pragma unroll
    for (int u = 0; u < kProdPairs; ++u) {
      const int64_t n = n0 + 2 * u + sub;
      row[u] = -1;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (n < a.n) {
        row[u] = __ldg(a.slot + n);
        if (row[u] >= a.num_rows) {
          if (hl == 0) raise_error(DSA_DEVERR_INDEX);
          row[u] = -1;
        }
        if (row[u] >= 0) raw[u] = __ldg(reinterpret_cast<const uint4*>(a.k + n * 128) + hl);
      }
    }
#pragma unroll
    for (int u = 0; u < kProdPairs; ++u) {
      const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
      float x[8];                                  // elements e = 8 hl + i
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
      }
      // butterflies over bits 0..2 of e inside the lane, then bits 3..6 (lane bits 0..3)
      // across the 16 lanes of the row: the lower index keeps a + b, the upper one a - b
#pragma unroll
      for (int m = 1; m < 8; m <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if ((i & m) == 0) {
            const float p = x[i], q = x[i + m];
            x[i] = p + q;
            x[i + m] = p - q;
          }
        }
      }
#pragma unroll
      for (int m = 1; m < 16; m <<= 1) {
        const bool upper = (hl & m) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float o = __shfl_xor_sync(0xFFFFFFFFu, x[i], m);
          x[i] = upper ? (o - x[i]) : (x[i] + o);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], norm);
      // group of 32 elements = 4 lanes
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
      for (int o = 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
      const int byte = amax > 0.f ? max(ef - 2, 0) : 0;
      const float inv = __uint_as_float((uint32_t)(254 - byte) << 23);   // 2^(127 - byte)
      uint32_t nib = 0;
      if (amax > 0.f) {                            // element 8 hl + i in nibble i
#pragma unroll
        for (int i = 0; i < 4; ++i)
          nib |= e2m1x2(__fmul_rn(x[2 * i + 1], inv), __fmul_rn(x[2 * i], inv)) << (8 * i);
        nib = positive_zeros8(nib);
      }
      // the 4 scale bytes of the row, from lanes 0, 4, 8, 12 of its half-warp
      uint32_t sbytes = 0;
#pragma unroll
      for (int g = 0; g < 4; ++g) sbytes |= (uint32_t)__shfl_sync(0xFFFFFFFFu, byte, 16 * sub + 4 * g) << (8 * g);
      if (row[u] >= 0) {
        reinterpret_cast<uint32_t*>(a.fp4 + row[u] * 64)[hl] = nib;
        if (hl == 0) *reinterpret_cast<uint32_t*>(a.scale + row[u] * 4) = sbytes;
      }
    }
  }
}

static int prod_grid(int64_t rows, int num_sms) {
  const int64_t warps = (rows + kProdRowsPerStep - 1) / kProdRowsPerStep;
  const int64_t blocks = (warps + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 8;      // 8 resident blocks of 256 threads per SM
  return (int)(blocks < cap ? blocks : cap);
}

cudaError_t launch_q_rope_quant(const uint16_t* q, const int32_t* positions, const float* cos_sin, int64_t max_pos,
                                int rope_dim, int64_t T, int H, uint8_t* codes, float* scale, int num_sms,
                                cudaStream_t stream) {
  const int64_t rows = T * H;
  if (rows <= 0) return cudaSuccess;
  QRopeArgs a{q, positions, cos_sin, max_pos, rope_dim, H, rows, codes, scale};
  q_rope_quant_kernel<<<prod_grid(rows, num_sms), 256, 0, stream>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_k_hadamard_mxfp4(const uint16_t* k, const int64_t* slot, int64_t n, uint8_t* fp4, uint8_t* scale,
                                    int64_t num_rows, int num_sms, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  KWriteArgs a{k, slot, n, num_rows, fp4, scale};
  k_hadamard_mxfp4_kernel<<<prod_grid(n, num_sms), 256, 0, stream>>>(a);
  note_launch();
  return cudaGetLastError();
}

DSA_DEFINE_TU_ERROR_ACCESSORS(producer)

}  // namespace dsa
