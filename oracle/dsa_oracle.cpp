// CPU oracle of the DeepSeek-V4 DSA indexer hot path -- TEST INFRASTRUCTURE ONLY.
//
// Plain, slow C++17: scalar loops in float64, one definition per function, written out
// in the order the problem states it.  Only the tests, the smoke check and the
// benchmark's CPU-baseline leg load this (through oracle/dsa_oracle.py); the CUDA
// library never does, and the two share no code, header, table or constant.  The only
// concession to speed is that independent query rows (or key ranges of one row) are
// handed to std::thread workers; every output element is computed by one thread with
// the same loops whatever the thread count.
//
// What each function computes, and the passage it follows:
//  * orc_indexer_logits -- the DSA indexer score (xkernels issue #27 "DSA indexer +
//    attention: validate/provide gfx942 forward path", comment 2 "What shipped"):
//    logits[t, j] = sum_h w[t, h] * relu(q[t, h, :] . k[j, :]), q [T, H, D], one shared
//    MQA key [K, D], per-head weights, optional per-query causal window.  Reading of the
//    window: query i of sequence b sits at p = L_b - next_n + i and sees key j iff
//    j <= p (non-causal: j < L_b).  Masked keys hold -inf (the same comment shows a -inf
//    literal as the masked value).  Keys may be bf16, OCP E4M3 with a per-row fp32 scale,
//    or rows of the paged mxfp4 cache (the fp8-q x fp4-k form the same issue names; its
//    comment 2 "Caveats / deferred" calls the packing an encoding detail, so the score is
//    taken over the dequantised keys).
//  * orc_topk -- per query the k largest scores (top-512 Flash / top-1024 Pro, issue
//    #27 "Context"), ordered by value descending then index ascending (the deterministic
//    "canonical" top-k sort of README "DeepSeek V4 Flash on a single AMD MI300X",
//    overlay table); -0.0 equals +0.0; -inf is never selected; short rows pad with -1.
//  * orc_e2m1 / orc_e8m0 / orc_mxfp4_gather -- the paged mxfp4 gather (xkernels issue
//    #28 "DeepSeek-V4 serving support -- tracking", comment 2 "What it does"): E2M1
//    nibbles with one E8M0 scale 2^(b-127) per 32 elements, 0xFF meaning a scale of 0,
//    positions read through a block table, dequantised to bf16, padded slots
//    (sel_pos < 0) -> zero rows.  The E2M1 value set {0, 0.5, 1, 1.5, 2, 3, 4, 6} is the
//    OCP Microscaling v1.0 definition, looked up by table here (the GPU decodes
//    arithmetically); the low nibble of byte i holds element 2i.
//  * orc_sparse_attn -- the sparse-attention consumer of the selection (ROCm/ATOM issue
//    #707, "CSA": "index-gather + online softmax + attn_sink bias").  Reading: for query
//    row t and head h, over the selected positions j of row t (sel_pos >= 0), the key and
//    value are the same dequantised cache row x_j (the latent of the paged mxfp4 cache
//    the gather reads); s_j = scale * q[t,h,:] . x_j; the head's sink logit joins the
//    softmax denominator only:  out[t,h,:] = sum_j e^(s_j - m) x_j / (sum_j e^(s_j - m)
//    + e^(sink_h - m)), m = max(max_j s_j, sink_h).  A row with no selected position
//    gives zeros.  The online (streaming) softmax is the GPU's way to compute this sum.
//  * orc_e4m3 -- OCP E4M3 (bias 7, no infinities, S.1111.111 = NaN, subnormals
//    m * 2^-9), the byte format README "DeepSeek V4 Flash on a single AMD MI300X"
//    ("FP8 format") contrasts with AMD's FNUZ variant; orc_e4m3_encode rounds to it
//    (nearest, ties to the even code, saturating at +-448 = the FP8_MAX the OCP path
//    uses, vllm PR #1 "Sparse-MLA bring-up on MI300X", "Root cause story" item 1).
//  * orc_q_rope_quant -- the indexer-Q producer ahead of the score (vllm PR #1, "Root
//    cause story" item 3: a fused RoPE + per-row FP8 quantisation of the indexer query
//    whose bytes the fp8 MQA-logits reader consumes).  Readings: RoPE rotates the
//    interleaved pairs (2i, 2i+1) of the first rope_dim dims of every head by the angle
//    whose cos / sin the caller's table holds for the token's position; the other dims
//    pass through; each (token, head) row is then quantised with scale = rowmax / 448
//    (1 for an all-zero row), code = E4M3(value / scale).  Arithmetic in fp32, each
//    product and sum rounded on its own (no fused multiply-add), because the codes are
//    integers decided by that arithmetic.
//  * orc_k_hadamard_mxfp4 -- the indexer-key compressor's write into the paged FP4
//    cache (ROCm/ATOM issue #707, "CSA": "CSA Indexer Compressor (head_dim=128,
//    Hadamard, FP4)"), read as: rotate each 128-dim key by the orthonormal
//    Walsh-Hadamard matrix (Sylvester order, entries +-1/sqrt(128)), then encode it in
//    the gather's mxfp4 layout by the OCP MX v1.0 conversion: per 32-element group
//    the shared exponent is floor(log2(amax)) - 2 (2 = the largest E2M1 exponent), the
//    E8M0 byte that exponent + 127 (clamped to 0..254; an all-zero group gets byte 0),
//    each element E2M1(value / 2^exponent) rounded to nearest, ties to the even code,
//    saturating at 6; low nibble = even element; written to the pool row its slot
//    names (slot < 0: skipped).  The rotation is computed in float64 and rounded to
//    fp32, the precision in which the codes are decided.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <utility>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// ------------------------------------------------------------------ decoding

// bf16 is the upper half of an IEEE binary32.
double bf16_value(uint16_t bits) {
  const uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// OCP E4M3: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
double e4m3_value(uint8_t c) {
  const int s = (c >> 7) & 1;
  const int e = (c >> 3) & 0xF;
  const int m = c & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  double mag;
  if (e == 0)
    mag = (m / 8.0) * std::ldexp(1.0, -6);             // subnormal
  else
    mag = (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);    // normal
  return s ? -mag : mag;
}

// E2M1 nibble s|e1 e0|m: magnitude by the OCP MX table, then the sign bit.
const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double e2m1_value(uint8_t nibble) {
  const double mag = kE2M1Magnitude[nibble & 7];
  return (nibble & 8) ? -mag : mag;
}

// E8M0 group scale: 2^(b - 127); the byte 0xFF means a scale of 0.
double e8m0_value(uint8_t b) { return b == 0xFF ? 0.0 : std::ldexp(1.0, static_cast<int>(b) - 127); }

// Round to bf16, nearest-even, through binary32 (exact for every value this oracle
// rounds: an E2M1 value times a power of two has at most two significant bits).
uint16_t bf16_bits_of(double x) {
  const float f = static_cast<float>(x);
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if (std::isnan(f)) return 0x7FC0;
  const uint32_t lsb = (u >> 16) & 1u;
  return static_cast<uint16_t>((static_cast<uint64_t>(u) + 0x7FFFu + lsb) >> 16);
}

// Element e of an mxfp4 row: nibble (e & 1) of byte e / 2, times the scale of group e / 32.
double mxfp4_element(const uint8_t* nib_row, const uint8_t* scale_row, int e) {
  const uint8_t byte = nib_row[e / 2];
  const uint8_t nibble = (e % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  return e2m1_value(nibble) * e8m0_value(scale_row[e / 32]);
}

// Nearest E4M3 code of a finite fp32 value: ties to the code with the even mantissa,
// magnitudes beyond 448 saturate to 448.  Found by rounding the value on the grid of
// its binade (subnormal spacing 2^-9 below 2^-6), then looking the rounded value up
// among the 256 codes.
uint8_t e4m3_encode(float xf) {
  const double x = static_cast<double>(xf);
  double a = std::fabs(x);
  if (a > 448.0) a = 448.0;
  double step;
  if (a < std::ldexp(1.0, -6)) {
    step = std::ldexp(1.0, -9);
  } else {
    int e;
    std::frexp(a, &e);                      // a = f * 2^e, f in [0.5, 1)
    step = std::ldexp(1.0, (e - 1) - 3);    // 3 mantissa bits below the leading one
  }
  const double q = a / step;                // exact: step is a power of two
  double r = std::floor(q);
  const double frac = q - r;
  if (frac > 0.5 || (frac == 0.5 && std::fmod(r, 2.0) != 0.0)) r += 1.0;
  const double v = r * step;                // <= 448: a <= 448 = 14 * 32 lies on the grid
  const bool neg = std::signbit(x);
  for (int c = 0; c < 128; ++c) {           // codes 0x00..0x7F are the non-negative values
    if (c == 0x7F) continue;                 // NaN
    if (e4m3_value(static_cast<uint8_t>(c)) == v) return static_cast<uint8_t>(neg ? (c | 0x80) : c);
  }
  return 0x7F;                               // not reached for finite inputs
}

// Nearest E2M1 code of a double value: ties to the code with the even mantissa bit,
// magnitudes beyond 6 saturate to 6.
uint8_t e2m1_encode(double x) {
  double a = std::fabs(x);
  if (a > 6.0) a = 6.0;
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double dc = std::fabs(kE2M1Magnitude[c] - a), db = std::fabs(kE2M1Magnitude[best] - a);
    if (dc < db || (dc == db && (c & 1) == 0)) best = c;
  }
  return static_cast<uint8_t>(best | (std::signbit(x) && best != 0 ? 8 : 0));
}

// ------------------------------------------------------------------ threads

// Runs fn(i) for i in [0, n) on up to `threads` workers (0: all hardware threads).
template <class F>
void parallel_for(int64_t n, int threads, F fn) {
  int nt = threads > 0 ? threads : static_cast<int>(std::thread::hardware_concurrency());
  if (nt < 1) nt = 1;
  if (n < nt) nt = static_cast<int>(n < 1 ? 1 : n);
  std::atomic<int64_t> next{0};
  auto work = [&]() {
    for (int64_t i = next.fetch_add(1); i < n; i = next.fetch_add(1)) fn(i);
  };
  std::vector<std::thread> pool;
  for (int w = 1; w < nt; ++w) pool.emplace_back(work);
  work();
  for (auto& th : pool) th.join();
}

// Storage kinds.
enum { kBF16 = 0, kE4M3 = 1, kMXFP4 = 2 };

}  // namespace

extern "C" {

int orc_threads_used(int threads) {
  const int hw = static_cast<int>(std::thread::hardware_concurrency());
  return threads > 0 ? threads : (hw > 0 ? hw : 1);
}

void orc_bf16(const uint16_t* bits, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(bits[i]);
}

void orc_e4m3(const uint8_t* codes, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

void orc_e2m1(const uint8_t* nibbles, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e2m1_value(nibbles[i] & 0xF);
}

void orc_e8m0(const uint8_t* bytes, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e8m0_value(bytes[i]);
}

void orc_bf16_round(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits_of(x[i]);
}

// rows x D/2 nibble bytes + rows x D/32 scale bytes -> rows x D values.
void orc_mxfp4_dequant(const uint8_t* nib, const uint8_t* scale, int64_t rows, int D, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int e = 0; e < D; ++e) out[r * D + e] = mxfp4_element(nib + r * (D / 2), scale + r * (D / 32), e);
}

// Indexer score of the query rows `rows` (nrows of them) into out [nrows, width].
//   q       [T, H, D] bf16 bits (q_kind 0) or E4M3 codes (q_kind 1); q_scale [T, H] (E4M3)
//   weights [T, H]
//   keys    k_kind 0: bf16 bits [num_rows, D]; 1: E4M3 codes [num_rows, D] with k_scale
//           [num_rows]; 2: mxfp4 nibble bytes [num_rows, D/2] with k_scale = E8M0 bytes
//           [num_rows, D/32]
//   (weights and scales are taken in float64: the fp32 values of the problem convert
//   exactly)
//   block_table [B, bt_stride] (NULL: contiguous keys of one sequence, key j = row j)
// Returns 0, or -1 when a key row falls outside the pool (the caller's inputs are wrong).
int orc_indexer_logits(const void* q, const double* q_scale, int q_kind, const double* weights, int H, int D,
                       const void* k_data, const void* k_scale, int k_kind, int64_t num_rows,
                       const int32_t* block_table, int64_t bt_stride, int block_size, int B, int next_n,
                       const int32_t* context_lens, int causal, const int64_t* rows, int64_t nrows, int64_t width,
                       double* out, int threads) {
  (void)B;
  std::atomic<int> bad{0};
  // Work unit: (row, 4096-key range), so one long row still uses every worker.
  const int64_t kChunk = 4096;
  const int64_t chunks = (width + kChunk - 1) / kChunk;
  parallel_for(nrows * (chunks > 0 ? chunks : 1), threads, [&](int64_t unit) {
    const int64_t r = unit / (chunks > 0 ? chunks : 1);
    const int64_t c = unit % (chunks > 0 ? chunks : 1);
    const int64_t t = rows[r];
    const int64_t b = t / next_n, i = t % next_n;
    const int64_t L = context_lens[b];
    int64_t visible = causal ? (L - next_n + i + 1) : L;
    if (visible < 0) visible = 0;
    if (visible > L) visible = L;
    // the query row, dequantised: qv[h][d]
    std::vector<double> qv(static_cast<size_t>(H) * D);
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < D; ++d) {
        const int64_t o = (t * H + h) * D + d;
        double v;
        if (q_kind == kBF16)
          v = bf16_value(static_cast<const uint16_t*>(q)[o]);
        else
          v = e4m3_value(static_cast<const uint8_t*>(q)[o]) * q_scale[t * H + h];
        qv[static_cast<size_t>(h) * D + d] = v;
      }
    std::vector<double> kv(D);
    const int64_t j0 = c * kChunk;
    const int64_t j1 = std::min(width, j0 + kChunk);
    for (int64_t j = j0; j < j1; ++j) {
      double* dst = out + r * width + j;
      if (j >= visible) {
        *dst = kNegInf;
        continue;
      }
      // physical row of logical key j
      int64_t row;
      if (block_table == nullptr) {
        row = j;
      } else {
        const int64_t blk = block_table[b * bt_stride + j / block_size];
        row = blk * block_size + j % block_size;
        if (blk < 0) row = -1;
      }
      if (row < 0 || row >= num_rows) {
        bad.store(1);
        *dst = std::numeric_limits<double>::quiet_NaN();
        continue;
      }
      // the key, dequantised
      for (int d = 0; d < D; ++d) {
        double v;
        if (k_kind == kBF16) {
          v = bf16_value(static_cast<const uint16_t*>(k_data)[row * D + d]);
        } else if (k_kind == kE4M3) {
          v = e4m3_value(static_cast<const uint8_t*>(k_data)[row * D + d]) *
              static_cast<const double*>(k_scale)[row];
        } else {
          const uint8_t* nib_row = static_cast<const uint8_t*>(k_data) + row * (D / 2);
          const uint8_t* scale_row = static_cast<const uint8_t*>(k_scale) + row * (D / 32);
          v = mxfp4_element(nib_row, scale_row, d);
        }
        kv[d] = v;
      }
      // sum over heads of weight * relu(dot)
      double logit = 0.0;
      for (int h = 0; h < H; ++h) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += qv[static_cast<size_t>(h) * D + d] * kv[d];
        const double relu = s > 0.0 ? s : 0.0;
        logit += weights[t * H + h] * relu;
      }
      *dst = logit + 0.0;     // -0.0 + 0.0 == +0.0
    }
  });
  return bad.load() ? -1 : 0;
}

// Top-k of each of R rows of `logits` [R, K] (value descending, index ascending);
// -inf is never selected, -0.0 ranks equal to +0.0.  idx [R, k] (-1 past the
// candidates), val [R, k] (-inf there).  Returns -1 if a row holds a NaN (outside the
// problem: ReLU of finite products and finite weights cannot produce one).
int orc_topk(const double* logits, int64_t R, int64_t K, int k, int32_t* idx, double* val, int threads) {
  std::atomic<int> nan_seen{0};
  parallel_for(R, threads, [&](int64_t r) {
    std::vector<std::pair<double, int64_t>> cand;
    for (int64_t j = 0; j < K; ++j) {
      const double v = logits[r * K + j];
      if (std::isnan(v)) nan_seen.store(1);
      if (v == kNegInf || std::isnan(v)) continue;
      cand.emplace_back(v + 0.0, j);      // canonical zero
    }
    std::sort(cand.begin(), cand.end(), [](const std::pair<double, int64_t>& a, const std::pair<double, int64_t>& b) {
      if (a.first != b.first) return a.first > b.first;   // larger value first
      return a.second < b.second;                         // then the smaller index
    });
    for (int s = 0; s < k; ++s) {
      if (s < static_cast<int64_t>(cand.size())) {
        idx[r * k + s] = static_cast<int32_t>(cand[s].second);
        val[r * k + s] = cand[s].first;
      } else {
        idx[r * k + s] = -1;
        val[r * k + s] = kNegInf;
      }
    }
  });
  return nan_seen.load() ? -1 : 0;
}

// out[t, s, :] = bf16(dequant(cache row of sel_pos[t, s])), zeros where sel_pos < 0.
// The sequence of row t is b = t / next_n; logical position pos lives in cache row
// (block_table[b, pos / block_size], pos % block_size).  kv_fp4 [num_blocks, block_size,
// D/2], kv_scale [num_blocks, block_size, D/32].  Returns -1 if a position maps outside
// the table or the pool.
int orc_mxfp4_gather(const uint8_t* kv_fp4, const uint8_t* kv_scale, int64_t num_blocks, int block_size, int D,
                     const int32_t* block_table, int64_t bt_stride, const int32_t* sel_pos, int64_t T, int next_n,
                     int k, uint16_t* out, int threads) {
  std::atomic<int> bad{0};
  parallel_for(T, threads, [&](int64_t t) {
    const int64_t b = t / next_n;
    for (int s = 0; s < k; ++s) {
      uint16_t* dst = out + (t * k + s) * D;
      const int64_t pos = sel_pos[t * k + s];
      if (pos < 0) {
        for (int e = 0; e < D; ++e) dst[e] = 0;
        continue;
      }
      const int64_t col = pos / block_size;
      const int64_t blk = col < bt_stride ? block_table[b * bt_stride + col] : -1;
      if (blk < 0 || blk >= num_blocks) {
        bad.store(1);
        for (int e = 0; e < D; ++e) dst[e] = 0;
        continue;
      }
      const int64_t row = blk * block_size + pos % block_size;
      for (int e = 0; e < D; ++e)
        dst[e] = bf16_bits_of(mxfp4_element(kv_fp4 + row * (D / 2), kv_scale + row * (D / 32), e));
    }
  });
  return bad.load() ? -1 : 0;
}

void orc_e2m1_encode(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e2m1_encode(x[i]);
}

void orc_e4m3_encode(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}

// q [T, H, D] bf16 bits, positions [T], cos_sin [max_pos, rope_dim] fp32 (per position:
// rope_dim / 2 cosines, then rope_dim / 2 sines) -> codes [T, H, D] E4M3, scale [T, H] fp32.
// Returns -1 if a position lies outside the table.
int orc_q_rope_quant(const uint16_t* q, const int32_t* positions, const float* cos_sin, int64_t max_pos,
                     int rope_dim, int64_t T, int H, int D, uint8_t* codes, float* scale, int threads) {
  std::atomic<int> bad{0};
  parallel_for(T * H, threads, [&](int64_t row) {
    const int64_t t = row / H;
    const int64_t pos = positions[t];
    if (pos < 0 || pos >= max_pos) {
      bad.store(1);
      for (int d = 0; d < D; ++d) codes[row * D + d] = 0;
      scale[row] = 0.0f;
      return;
    }
    std::vector<float> y(D);
    for (int d = 0; d < D; ++d) y[d] = static_cast<float>(bf16_value(q[row * D + d]));
    const int half = rope_dim / 2;
    for (int i = 0; i < half; ++i) {
      const float x0 = y[2 * i], x1 = y[2 * i + 1];
      const float c = cos_sin[pos * rope_dim + i], s = cos_sin[pos * rope_dim + half + i];
      const float p0 = x0 * c, p1 = x1 * s, p2 = x0 * s, p3 = x1 * c;
      y[2 * i] = p0 - p1;
      y[2 * i + 1] = p2 + p3;
    }
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) amax = std::max(amax, std::fabs(y[d]));
    const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    scale[row] = sc;
    for (int d = 0; d < D; ++d) codes[row * D + d] = e4m3_encode(y[d] / sc);
  });
  return bad.load() ? -1 : 0;
}

// k [N, D] bf16 bits, slot [N] (pool row or < 0) -> kv_fp4 [num_rows, D/2],
// kv_scale [num_rows, D/32] at the slots' rows.  D must be a power of two.
// Returns -1 if a slot lies outside the pool.
int orc_k_hadamard_mxfp4(const uint16_t* k, const int64_t* slot, int64_t N, int D, uint8_t* kv_fp4,
                         uint8_t* kv_scale, int64_t num_rows, int threads) {
  std::atomic<int> bad{0};
  const double norm = 1.0 / std::sqrt(static_cast<double>(D));
  parallel_for(N, threads, [&](int64_t n) {
    const int64_t row = slot[n];
    if (row < 0) return;
    if (row >= num_rows) {
      bad.store(1);
      return;
    }
    std::vector<double> x(D);
    std::vector<float> y(D);
    for (int d = 0; d < D; ++d) x[d] = bf16_value(k[n * D + d]);
    // y_i = sum_j H[i][j] x_j / sqrt(D), H[i][j] = (-1)^popcount(i & j) (Sylvester order)
    for (int i = 0; i < D; ++i) {
      double acc = 0.0;
      for (int j = 0; j < D; ++j) {
        const int sign = __builtin_popcount(static_cast<unsigned>(i & j)) & 1;
        acc += sign ? -x[j] : x[j];
      }
      y[i] = static_cast<float>(acc * norm);
    }
    for (int g = 0; g < D / 32; ++g) {
      float amax = 0.0f;
      for (int e = 0; e < 32; ++e) amax = std::max(amax, std::fabs(y[g * 32 + e]));
      int sexp = 0;                                  // shared exponent
      uint8_t byte = 0;
      if (amax > 0.0f) {
        int e2;
        std::frexp(static_cast<double>(amax), &e2);  // amax = f * 2^e2, f in [0.5, 1)
        sexp = (e2 - 1) - 2;                         // floor(log2(amax)) - 2
        int b = sexp + 127;
        if (b < 0) b = 0;
        if (b > 254) b = 254;
        byte = static_cast<uint8_t>(b);
        sexp = b - 127;
      }
      kv_scale[row * (D / 32) + g] = byte;
      for (int e = 0; e < 32; e += 2) {
        uint8_t lo = 0, hi = 0;
        if (amax > 0.0f) {
          lo = e2m1_encode(std::ldexp(static_cast<double>(y[g * 32 + e]), -sexp));
          hi = e2m1_encode(std::ldexp(static_cast<double>(y[g * 32 + e + 1]), -sexp));
        }
        kv_fp4[row * (D / 2) + (g * 32 + e) / 2] = static_cast<uint8_t>(lo | (hi << 4));
      }
    }
  });
  return bad.load() ? -1 : 0;
}

// q [T, H, D] bf16 bits, sel [T, k], cache kv_fp4 [num_blocks, block_size, D/2] +
// kv_scale [num_blocks, block_size, D/32], block_table [B, bt_stride], sink [H] ->
// out [T, H, D] (float64).  Returns -1 if a selected position maps outside the cache.
int orc_sparse_attn(const uint16_t* q, const int32_t* sel, int64_t T, int H, int D, int k, const uint8_t* kv_fp4,
                    const uint8_t* kv_scale, int64_t num_blocks, int block_size, const int32_t* block_table,
                    int64_t bt_stride, int next_n, const double* sink, double scale, double* out, int threads) {
  std::atomic<int> bad{0};
  parallel_for(T, threads, [&](int64_t t) {
    const int64_t b = t / next_n;
    // the row's selected keys / values, dequantised
    std::vector<double> x;
    int n = 0;
    for (int s = 0; s < k; ++s) {
      const int64_t pos = sel[t * k + s];
      if (pos < 0) continue;
      const int64_t page = pos / block_size;
      const int64_t block = page < bt_stride ? block_table[b * bt_stride + page] : -1;
      if (block < 0 || block >= num_blocks) {
        bad.store(1);
        continue;
      }
      const int64_t crow = block * block_size + pos % block_size;
      for (int e = 0; e < D; ++e) x.push_back(mxfp4_element(kv_fp4 + crow * (D / 2), kv_scale + crow * (D / 32), e));
      ++n;
    }
    for (int h = 0; h < H; ++h) {
      double* o = out + (t * H + h) * D;
      for (int e = 0; e < D; ++e) o[e] = 0.0;
      if (n == 0) continue;
      std::vector<double> sc(n);
      double m = sink[h];
      for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int e = 0; e < D; ++e) dot += bf16_value(q[(t * H + h) * D + e]) * x[(size_t)j * D + e];
        sc[j] = scale * dot;
        m = std::max(m, sc[j]);
      }
      double denom = std::exp(sink[h] - m);
      for (int j = 0; j < n; ++j) {
        const double p = std::exp(sc[j] - m);
        denom += p;
        for (int e = 0; e < D; ++e) o[e] += p * x[(size_t)j * D + e];
      }
      for (int e = 0; e < D; ++e) o[e] /= denom;
    }
  });
  return bad.load() ? -1 : 0;
}

}  // extern "C"
