// Producers around the indexer score (sm_103a): the indexer-query RoPE + per-row FP8
// quantisation ahead of it, and the indexer-key Hadamard rotation + mxfp4 write into
// the paged cache that the score (FP4-key form) and the gather read.
//
// Indexer-Q producer (vllm PR #1 "Sparse-MLA bring-up on MI300X", "Root cause story"
// item 3: a fused RoPE + FP8 quantisation of the indexer query, FP8_MAX = 448 on the OCP
// path).  One warp per (token, head) row of 128 dims, 4 dims per lane: the interleaved
// pairs (2i, 2i+1) of the first rope_dim dims turn by the table's cos / sin for the
// token's position, the row's largest magnitude gives scale = amax / 448, and each dim
// becomes E4M3(value / scale) (nearest even, saturating).  Every product and sum is
// rounded on its own (no contraction into FMAs): the codes are integers decided by that
// fp32 arithmetic.
//
// Indexer-key writer (ROCm/ATOM issue #707, "CSA": "CSA Indexer Compressor
// (head_dim=128, Hadamard, FP4)").  One warp per key of 128 dims, 4 per lane: a
// 128-point Walsh-Hadamard transform (Sylvester order; two butterfly stages inside a
// lane, five across lanes by shuffles) scaled by 1/sqrt(128), then the OCP MX encoding
// of the gather's layout: per 32-element group (8 lanes) the E8M0 byte is
// max(exponent field of amax - 2, 0) (= floor(log2 amax) - 2 + 127), each element the
// nearest E2M1 code of value / 2^(byte - 127) (ties to the even code, saturating at 6, by
// the hardware conversion; zero results +0), packed two per byte, low nibble = even element.
//
// Both are HBM-bound streams (a few hundred bytes per row); loads for several rows are
// issued before any of them is used.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace dsa {

constexpr int kProdRowsPerWarp = 4;

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
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int d0 = lane * 4;                       // this lane's dims d0 .. d0 + 3
  const bool rotate = d0 < a.rope_dim;           // rope_dim is a multiple of 4
  const int half = a.rope_dim >> 1;
  for (int64_t r0 = warp * kProdRowsPerWarp; r0 < a.rows; r0 += nwarps * kProdRowsPerWarp) {
    uint2 raw[kProdRowsPerWarp];
    float4 cs[kProdRowsPerWarp];                 // cos(pair 2l), cos(2l+1), sin(2l), sin(2l+1)
    bool ok[kProdRowsPerWarp];
#pragma unroll
    for (int u = 0; u < kProdRowsPerWarp; ++u) {
      const int64_t r = r0 + u;
      raw[u] = make_uint2(0u, 0u);
      cs[u] = make_float4(1.f, 1.f, 0.f, 0.f);
      ok[u] = false;
      if (r < a.rows) {
        raw[u] = __ldg(reinterpret_cast<const uint2*>(a.q + r * 128) + lane);
        const int64_t pos = __ldg(a.positions + r / a.H);
        ok[u] = pos >= 0 && pos < a.max_pos;
        if (ok[u] && rotate) {
          const float* row = a.cos_sin + pos * a.rope_dim;
          const float2 c = __ldg(reinterpret_cast<const float2*>(row + (d0 >> 1)));
          const float2 s = __ldg(reinterpret_cast<const float2*>(row + half + (d0 >> 1)));
          cs[u] = make_float4(c.x, c.y, s.x, s.y);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kProdRowsPerWarp; ++u) {
      const int64_t r = r0 + u;
      float y[4] = {bf16_bits_to_f32(raw[u].x & 0xFFFFu), bf16_bits_to_f32(raw[u].x >> 16),
                    bf16_bits_to_f32(raw[u].y & 0xFFFFu), bf16_bits_to_f32(raw[u].y >> 16)};
      if (rotate) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const float x0 = y[2 * p], x1 = y[2 * p + 1];
          const float c = p ? cs[u].y : cs[u].x, s = p ? cs[u].w : cs[u].z;
          y[2 * p] = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
          y[2 * p + 1] = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
        }
      }
      float amax = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
      uint32_t packed = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(y[e], sc), __NV_SATFINITE, __NV_E4M3);
        packed |= (uint32_t)c << (8 * e);
      }
      if (r < a.rows) {
        if (!ok[u]) {
          packed = 0;
          if (lane == 0) raise_error(DSA_DEVERR_INDEX);
        }
        reinterpret_cast<uint32_t*>(a.codes + r * 128)[lane] = packed;
        if (lane == 0) a.scale[r] = ok[u] ? sc : 0.f;
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

// Clears the sign of every nibble of `nib` (4 nibbles) whose magnitude is 0: a value that
// rounds to zero is written as +0.
__device__ __forceinline__ uint32_t positive_zeros4(uint32_t nib) {
  const uint32_t mag = nib & 0x7777u;
  const uint32_t nz = (mag | (mag >> 1) | (mag >> 2)) & 0x1111u;
  return nib & ((nz << 3) | 0x7777u);
}

__global__ void __launch_bounds__(256) k_hadamard_mxfp4_kernel(const KWriteArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const float norm = 0.08838834764831845f;       // 1 / sqrt(128), rounded to fp32
  for (int64_t n0 = warp * kProdRowsPerWarp; n0 < a.n; n0 += nwarps * kProdRowsPerWarp) {
    uint2 raw[kProdRowsPerWarp];
    int64_t row[kProdRowsPerWarp];
#pragma unroll
    for (int u = 0; u < kProdRowsPerWarp; ++u) {
      const int64_t n = n0 + u;
      row[u] = -1;
      raw[u] = make_uint2(0u, 0u);
      if (n < a.n) {
        row[u] = __ldg(a.slot + n);
        if (row[u] >= a.num_rows) {
          if (lane == 0) raise_error(DSA_DEVERR_INDEX);
          row[u] = -1;
        }
        if (row[u] >= 0) raw[u] = __ldg(reinterpret_cast<const uint2*>(a.k + n * 128) + lane);
      }
    }
#pragma unroll
    for (int u = 0; u < kProdRowsPerWarp; ++u) {
      float x[4] = {bf16_bits_to_f32(raw[u].x & 0xFFFFu), bf16_bits_to_f32(raw[u].x >> 16),
                    bf16_bits_to_f32(raw[u].y & 0xFFFFu), bf16_bits_to_f32(raw[u].y >> 16)};
      // element index e = 4 * lane + i; butterflies over bit 0, 1 (in the lane), then
      // bits 2..6 (lane bits 0..4): partner keeps a + b at the lower index, a - b above
      {
        const float a0 = x[0] + x[1], a1 = x[0] - x[1], a2 = x[2] + x[3], a3 = x[2] - x[3];
        x[0] = a0 + a2;
        x[1] = a1 + a3;
        x[2] = a0 - a2;
        x[3] = a1 - a3;
      }
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float o = __shfl_xor_sync(0xFFFFFFFFu, x[i], m);
          x[i] = upper ? (o - x[i]) : (x[i] + o);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = __fmul_rn(x[i], norm);
      // group of 32 elements = 8 lanes
      float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
      const int byte = amax > 0.f ? max(ef - 2, 0) : 0;
      const float inv = __uint_as_float((uint32_t)(254 - byte) << 23);   // 2^(127 - byte)
      uint32_t nib = 0;
      if (amax > 0.f)                            // element 4 lane + i in nibble i
        nib = positive_zeros4(e2m1x2(__fmul_rn(x[1], inv), __fmul_rn(x[0], inv)) |
                              (e2m1x2(__fmul_rn(x[3], inv), __fmul_rn(x[2], inv)) << 8));
      // the 4 scale bytes of the row, from lanes 0, 8, 16, 24
      uint32_t sbytes = 0;
#pragma unroll
      for (int g = 0; g < 4; ++g) sbytes |= (uint32_t)__shfl_sync(0xFFFFFFFFu, byte, 8 * g) << (8 * g);
      if (row[u] >= 0) {
        reinterpret_cast<uint16_t*>(a.fp4 + row[u] * 64)[lane] = (uint16_t)nib;
        if (lane == 0) *reinterpret_cast<uint32_t*>(a.scale + row[u] * 4) = sbytes;
      }
    }
  }
}

static int prod_grid(int64_t rows, int num_sms) {
  const int64_t warps = (rows + kProdRowsPerWarp - 1) / kProdRowsPerWarp;
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
