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
//  * orc_e4m3 -- OCP E4M3 (bias 7, no infinities, S.1111.111 = NaN, subnormals
//    m * 2^-9), the byte format README "DeepSeek V4 Flash on a single AMD MI300X"
//    ("FP8 format") contrasts with AMD's FNUZ variant.
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

}  // extern "C"
