// Sparse attention over the indexer's selection, reading the paged mxfp4 cache directly
// (ROCm/ATOM issue #707, "CSA": "index-gather + online softmax + attn_sink bias").
// Reading of the step: for query row t and head h, over the selected positions j of row t
// (sel_pos >= 0) the key and the value are the same dequantised cache row x_j;
// s_j = scale * q[t,h,:] . x_j, and the head's sink logit joins the softmax denominator
// only:  out[t,h,:] = sum_j e^(s_j - m) x_j / (sum_j e^(s_j - m) + e^(sink_h - m)).
//
// One CTA per query row: 64 heads x 128 dims, the selection in tiles of 128 rows.
//  * Four converter / softmax warps.  Thread j owns row j of each tile: it resolves the
//    row's cache position (block table), loads its 64 nibble bytes and 4 scale bytes,
//    decodes them to bf16 (exact: every E2M1 x E8M0 value is a bf16 value; by byte
//    permutation, no shared table) into the
//    tile X [128 rows][128 dims] (K-major, 128-byte swizzle).  The next tile's bytes are
//    in flight while the current tile's softmax runs.
//  * One MMA thread, three tcgen05 products per tile, accumulators in tensor memory:
//      S^T [128 rows, 64 heads]  = X . Q^T          (A = X K-major, B = Q K-major)
//      O^T [128 dims, 64 heads] += X^T . P^T        (A = the same X tile read dims-major,
//                                                    B = P [rows][heads] read heads-major)
//      L   [128 x 64 heads]     += 1 . P^T          (A = a ones tile: every lane of L
//                                                    holds the column sums of P)
//    The transposed form keeps every product at M = 128 with the 64 heads as N; the
//    score tile's TMEM lane is the row the thread decoded, and the output's lane is a dim.
//  * Softmax in base 2 (scores times scale * log2 e).  Per head, the tile maximum comes
//    from a butterfly across the warp and a pass over the four warps' results; the
//    running maximum starts at the sink logit and moves only when a tile's maximum
//    exceeds it by more than 8 (so P <= 2^8 in bf16); O and L are then rescaled in tensor
//    memory.  P is rounded to bf16 once and the same values feed O and L, so numerator
//    and denominator use identical weights.
// Every selected slot's cache row is resolved (selection, then block table) into shared
// memory when the CTA starts, so the per-tile loads depend on nothing in flight.
// Tensor memory: S double-buffered (2 x 64 columns), O and L (64 each): 256 columns;
// 101 KB of shared memory + 4 B per selected slot: two CTAs per SM up to top-2048.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace dsa {

namespace {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kTile = 128;
constexpr int kGroup = 128;                 // converter / softmax threads
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;               // base-2 headroom before the running max moves

// shared-memory layout (from a 1024-byte aligned base)
constexpr uint32_t kQOff = 0;               // Q [64 heads][128 dims] bf16, two 8 KB K chunks
constexpr uint32_t kXOff = 16384;           // X tiles [2][2 K chunks][128 rows][128 B]
constexpr uint32_t kXBytes = 32768;
constexpr uint32_t kPOff = kXOff + 2 * kXBytes;        // P [128 rows][64 heads] bf16
constexpr uint32_t kOnesOff = kPOff + 16384;           // two 1 KB swizzle atoms of bf16 1.0
constexpr uint32_t kRedOff = kOnesOff + 2048;          // per-warp head maxima [4][64]
constexpr uint32_t kMOff = kRedOff + 1024;             // running max [64]
constexpr uint32_t kFacOff = kMOff + 256;              // this tile's rescale factors [64]
constexpr uint32_t kSinkOff = kFacOff + 256;           // sink logits, base 2 [64]
constexpr uint32_t kFlagOff = kSinkOff + 256;          // rescale stamp, abort, TMEM base
constexpr uint32_t kBarOff = kFlagOff + 16;
constexpr int kNumBars = 12;
constexpr uint32_t kRowsOff = kBarOff + 8 * kNumBars;  // cache row of every selected slot [ntiles * 128]
constexpr int kMaxTopk = 16384;

// dynamic shared memory for a selection of k slots (+ alignment slack)
__host__ __device__ constexpr size_t attn_smem_bytes(int k) {
  return kRowsOff + (size_t)((k + 127) / 128) * 128 * 4 + 1024;
}

constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;               // S buffers at 0 and 64
constexpr uint32_t kColO = 128;
constexpr uint32_t kColL = 192;

// instruction descriptors: bf16 x bf16 -> fp32, M = 128, N = 64; bit 15 / 16 mark A / B
// as MN-major (the contiguous dimension is M / N instead of K)
constexpr uint32_t kIdescS = idesc_bf16(128, kHeads);
constexpr uint32_t kIdescO = idesc_bf16(128, kHeads) | (1u << 15) | (1u << 16);
constexpr uint32_t kIdescL = idesc_bf16(128, kHeads) | (1u << 16);

struct AttnArgs {
  const uint16_t* q;         // [T, 64, 128] bf16
  const int32_t* sel;        // [T, k]
  int k;
  const uint8_t* fp4;        // [num_blocks * bs, 64]
  const uint8_t* scale;      // [num_blocks * bs, 4]
  int64_t num_blocks;
  int bs;
  const int32_t* table;      // [B, bt_stride]
  int64_t bt_stride;
  int next_n;
  const float* sink;         // [64]
  float scale_log2;          // softmax scale * log2 e
  float* out;                // [T, 64, 128] fp32
  int split;                 // CTAs per query row (a cluster; 1, 2 or 4)
};

// Shared-memory descriptor with explicit byte offsets (128-byte swizzle).  K-major: SBO =
// stride of 8-row groups.  MN-major: LBO = stride of 64-element atoms along M / N, SBO =
// stride of 8-row groups along K.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// 32 consecutive 32-bit columns of the thread's own TMEM lane: load (completed by
// tcgen05.wait::ld) and store (completed by tcgen05.wait::st).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "{\n tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n tcgen05.wait::ld.sync.aligned;\n}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Named barrier over the 128 group threads that also ANDs a predicate across them.
__device__ __forceinline__ bool group_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The raw bytes of one selected row (or none).
struct RawRow {
  uint4 w[4];
  uint32_t sc;
  bool valid;
};

// Cache row of selected position pos of query row t (-1: padded, or dropped with
// DSA_DEVERR_INDEX when the block table does not map it into the cache).
__device__ __forceinline__ int32_t resolve_row(const AttnArgs& a, int64_t t, int32_t pos) {
  if (pos < 0) return -1;
  const int64_t b = t / a.next_n;
  const int32_t page = pos / a.bs;
  if (page < a.bt_stride) {
    const int32_t blk = __ldg(a.table + b * a.bt_stride + page);
    if (blk >= 0 && blk < a.num_blocks) return blk * a.bs + pos % a.bs;
  }
  raise_error(DSA_DEVERR_INDEX);
  return -1;
}

__device__ __forceinline__ RawRow load_row(const AttnArgs& a, int32_t row) {
  RawRow r;
  r.valid = row >= 0;
  r.sc = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < 4; ++i) r.w[i] = make_uint4(0u, 0u, 0u, 0u);
  if (row < 0) return r;
  const uint4* src = reinterpret_cast<const uint4*>(a.fp4 + (int64_t)row * 64);
#pragma unroll
  for (int i = 0; i < 4; ++i) r.w[i] = __ldg(src + i);
  r.sc = __ldg(reinterpret_cast<const uint32_t*>(a.scale + (int64_t)row * 4));
  return r;
}

// Row j of an X tile: 128 bf16 dims, dims 64 c .. 64 c + 63 in K chunk c (16 KB apart),
// 16-byte piece p of row j at j * 128 + ((p ^ (j & 7)) << 4).
__device__ __forceinline__ void decode_row(const RawRow& r, uint8_t* tile, int j) {
  uint8_t* dst = tile + j * 128;
  // all 16 pieces are decoded before any is stored: a store between two table reads would
  // keep the compiler from issuing the reads together (it cannot tell them apart)
  auto put = [&](auto decode) {
    uint4 o[16];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t b = (r.sc >> (8 * g)) & 0xFFu;
      const uint32_t words[4] = {r.w[g].x, r.w[g].y, r.w[g].z, r.w[g].w};
#pragma unroll
      for (int w = 0; w < 4; ++w) o[4 * g + w] = decode(words[w], b);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int pc = ((i >> 2) & 1) * 4 + (i & 3);
      *reinterpret_cast<uint4*>(dst + (i >> 3) * 16384 + ((pc ^ (j & 7)) << 4)) = o[i];
    }
  };
  if (!r.valid)
    put([](uint32_t, uint32_t) { return make_uint4(0u, 0u, 0u, 0u); });
  else if (!e8m0_word_off_table(r.sc))
    put([](uint32_t w, uint32_t b) { return decode8_perm(w, e2m1_bytes(b)); });
  else
    put([](uint32_t w, uint32_t b) { return decode8_exact(w, b); });
}

// Thread-block cluster: a barrier over every thread of the cluster (release / acquire), and
// a load from the same shared-memory variable of another CTA of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_peer(const float* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__global__ void __launch_bounds__(32 + kGroup, 2) sparse_attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* q_s = sm + kQOff;
  uint8_t* x_s = sm + kXOff;
  uint8_t* p_s = sm + kPOff;
  float* red = reinterpret_cast<float*>(sm + kRedOff);
  float* mrun = reinterpret_cast<float*>(sm + kMOff);
  float* fac = reinterpret_cast<float*>(sm + kFacOff);
  float* sink2 = reinterpret_cast<float*>(sm + kSinkOff);
  int* flags = reinterpret_cast<int*>(sm + kFlagOff);    // [0] rescale stamp, [1] abort, [2] TMEM base
  const uint32_t bar0 = smem_u32(sm + kBarOff);
  const uint32_t qfull = bar0, pfull = bar0 + 8, pfree = bar0 + 16, drain = bar0 + 24;
  auto xfull = [&](int b) { return bar0 + 32 + 8 * b; };
  auto xfree = [&](int b) { return bar0 + 48 + 8 * b; };
  auto sfull = [&](int b) { return bar0 + 64 + 8 * b; };
  auto sfree = [&](int b) { return bar0 + 80 + 8 * b; };
  volatile int* abort_flag = flags + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.split;                          // the cluster of CTAs sharing query row t
  const int64_t t = blockIdx.x / S;
  const int rank = (int)(blockIdx.x % S);         // = the CTA's rank in its cluster
  const int nall = (a.k + kTile - 1) / kTile;
  const int tile0 = (int)((int64_t)nall * rank / S);          // this CTA's tiles of the selection
  const int ntiles = (int)((int64_t)nall * (rank + 1) / S) - tile0;
  const unsigned long long limit = wait_limit_ns();

  if (threadIdx.x == 0) {
    mbar_init(qfull, kGroup);
    mbar_init(pfull, kGroup);
    mbar_init(pfree, 1);
    mbar_init(drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(xfull(b), kGroup);
      mbar_init(xfree(b), 1);
      mbar_init(sfull(b), 1);
      mbar_init(sfree(b), 4);
    }
    flags[0] = 0;
    flags[1] = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(flags + 2), kTmemCols);
  if (warp > 0) {
    const int gt = threadIdx.x - 32;
    // the ones tile: 2 KB of bf16 1.0
    reinterpret_cast<uint4*>(sm + kOnesOff)[gt] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)flags[2];
  grid_dependency_wait();               // q, the selection and the sinks may come from the kernel before

  if (warp == 0) {
    // ================================ MMA issue ================================
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(qfull, 0u, limit, abort_flag);
      const uint32_t qa = smem_u32(q_s), pa = smem_u32(p_s), ones = smem_u32(sm + kOnesOff);
      for (int i = 0; ok && i <= ntiles; ++i) {
        if (i < ntiles) {                         // S^T of tile i
          const int b = i & 1;
          const uint32_t u = (uint32_t)(i >> 1) & 1u;
          if (!(ok = mbar_wait(xfull(b), u, limit, abort_flag) && mbar_wait(sfree(b), u ^ 1u, limit, abort_flag)))
            break;
          tc_fence_after();
          const uint32_t xa = smem_u32(x_s + b * kXBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u;
            const uint32_t qoff = (uint32_t)(kk >> 2) * 8192u + (uint32_t)(kk & 3) * 32u;
            mma_bf16(tmem + kColS + 64u * (uint32_t)b, desc_sw128(xa + off, 16u, 1024u),
                     desc_sw128(qa + qoff, 16u, 1024u), kIdescS, kk > 0 ? 1u : 0u);
          }
          mma_commit(sfull(b));
        }
        if (i > 0) {                              // O^T and L of tile i - 1
          const int j = i - 1, b = j & 1;
          if (!(ok = mbar_wait(pfull, (uint32_t)j & 1u, limit, abort_flag))) break;
          tc_fence_after();
          const uint32_t xa = smem_u32(x_s + b * kXBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {        // 16 selected rows per step
            const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
            const uint64_t pdesc = desc_sw128(pa + (uint32_t)kk * 2048u, 1024u, 1024u);
            mma_bf16(tmem + kColO, desc_sw128(xa + (uint32_t)kk * 2048u, 16384u, 1024u), pdesc, kIdescO, acc);
            const uint32_t ooff = (uint32_t)(kk >> 2) * 1024u + (uint32_t)(kk & 3) * 32u;
            mma_bf16(tmem + kColL, desc_sw128(ones + ooff, 16u, 0u), pdesc, kIdescL, acc);
          }
          mma_commit(xfree(b));
          mma_commit(pfree);
        }
      }
      if (!ok) {
        raise_error(DSA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      mma_commit(drain);                          // everything issued has completed
      mbar_wait(drain, 0u, kCleanupWaitNs, nullptr);
    }
    __syncwarp();
  } else {
    // ============================ converters + softmax ============================
    const int gt = threadIdx.x - 32;
    const int j = 32 * (warp & 3) + lane;         // TMEM lane: tile row (S^T) and dim (O^T)
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    float* orow = a.out + t * (kHeads * kDim);
    float* opart = reinterpret_cast<float*>(x_s);   // split rows: this CTA's O [64 heads][128 dims]
    float* lpart = red;                              // and its row sums L [64]
    if (ntiles == 0) {
      if (S == 1) {
        for (int h = 0; h < kHeads; ++h) orow[h * kDim + j] = 0.f;
      } else {
        for (int h = 0; h < kHeads; ++h) opart[h * kDim + j] = 0.f;
        if (gt < kHeads) {
          const float s2 = __ldg(a.sink + gt) * kLog2e;
          sink2[gt] = s2;
          mrun[gt] = s2;
          lpart[gt] = 0.f;
        }
      }
    } else {
      // the Q tile (K-major, 128-byte swizzle) and the sinks
      const uint4* qrow = reinterpret_cast<const uint4*>(a.q + t * (kHeads * kDim));
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int idx = gt + kGroup * r;          // 16-byte piece of the 64 x 256-byte tile
        const int h = idx >> 4, p16 = idx & 15;
        const uint4 v = __ldg(qrow + idx);
        *reinterpret_cast<uint4*>(q_s + (p16 >> 3) * 8192 + h * 128 + (((p16 & 7) ^ (h & 7)) << 4)) = v;
      }
      if (gt < kHeads) {
        const float s2 = __ldg(a.sink + gt) * kLog2e;
        sink2[gt] = s2;
        mrun[gt] = s2;                            // the running max starts at the sink logit
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(qfull);

      // every selected slot's cache row, resolved once: the positions first (all loads in
      // flight together), then their block-table entries
      int32_t* rows_s = reinterpret_cast<int32_t*>(sm + kRowsOff);
      for (int m0 = 0; m0 < ntiles; m0 += 8) {
        int32_t pos[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int slot = (tile0 + m0 + u) * kTile + j;
          pos[u] = (m0 + u < ntiles && slot < a.k) ? __ldg(a.sel + t * a.k + slot) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (m0 + u < ntiles) rows_s[(m0 + u) * kTile + j] = resolve_row(a, t, pos[u]);
      }

      bool ok = true;
      RawRow raw = load_row(a, rows_s[j]);
      decode_row(raw, x_s, j);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(xfull(0));
      if (ntiles > 1) raw = load_row(a, rows_s[kTile + j]);

      for (int i = 0; i < ntiles; ++i) {
        // scores of tile i (read twice from tensor memory: for the maximum, then for P)
        const int b = i & 1;
        const bool live = rows_s[i * kTile + j] >= 0;
        const uint32_t scol = tl + kColS + 64u * (uint32_t)b;
        ok &= mbar_wait(sfull(b), (uint32_t)(i >> 1) & 1u, limit, abort_flag);
        tc_fence_after();
        {
          uint32_t sv[64];
          tmem_ld64_issue(scol, sv);
          tmem_ld64_wait(sv);
          // per-head maximum over the warp's 32 rows, 32 heads at a time: a butterfly that
          // halves the values each step leaves lane l with head 32 hh + l
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float m16[16];
            {
              const bool hi = (lane & 16) != 0;
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float lo_v = live ? __uint_as_float(sv[32 * hh + e]) * a.scale_log2 : -INFINITY;
                const float hi_v = live ? __uint_as_float(sv[32 * hh + e + 16]) * a.scale_log2 : -INFINITY;
                m16[e] = fmaxf(hi ? hi_v : lo_v, __shfl_xor_sync(0xFFFFFFFFu, hi ? lo_v : hi_v, 16));
              }
            }
#pragma unroll
            for (int half = 8; half >= 1; half >>= 1) {
              const bool hi = (lane & half) != 0;
#pragma unroll
              for (int e = 0; e < half; ++e) {
                const float keep = hi ? m16[e + half] : m16[e];
                const float send = hi ? m16[e] : m16[e + half];
                m16[e] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, half));
              }
            }
            red[(warp & 3) * 64 + 32 * hh + lane] = m16[0];
          }
        }
        if (!(ok = group_all(ok))) break;
        if (gt < kHeads) {
          const float mt = fmaxf(fmaxf(red[gt], red[64 + gt]), fmaxf(red[128 + gt], red[192 + gt]));
          const float mo = mrun[gt];
          const float mn = mt > mo + kLazy ? mt : mo;
          const float f = mn == mo ? 1.f : ex2(mo - mn);
          fac[gt] = f;
          mrun[gt] = mn;
          if (f != 1.f) flags[0] = i + 1;
        }
        if (!(ok = group_all(ok))) break;
        // decode tile i + 1 into the buffer of tile i - 1: its products were issued with
        // tile i - 1's P, before this tile's maximum was taken, so they are done or nearly
        if (i + 1 < ntiles) {
          const int T = i + 1, xb = T & 1;
          ok &= mbar_wait(xfree(xb), ((uint32_t)(T >> 1) & 1u) ^ 1u, limit, abort_flag);
          decode_row(raw, x_s + xb * kXBytes, j);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(xfull(xb));
          if (i + 2 < ntiles) raw = load_row(a, rows_s[(i + 2) * kTile + j]);
        }
        // P (and the rescale of O and L) once the products of tile i - 1 are done
        if (i > 0) ok &= mbar_wait(pfree, (uint32_t)(i - 1) & 1u, limit, abort_flag);
        tc_fence_after();
        if (i > 0 && flags[0] == i + 1) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {             // O heads 0-31, 32-63, then L
            const uint32_t col = (c < 2 ? kColO : kColL) + 32u * (uint32_t)(c & 1);
            uint32_t acc[32];
            tmem_ld32(tl + col, acc);
#pragma unroll
            for (int h = 0; h < 32; ++h) acc[h] = __float_as_uint(__uint_as_float(acc[h]) * fac[32 * (c & 1) + h]);
            tmem_st32(tl + col, acc);
          }
          tmem_wait_st();
        }
        {
          uint32_t sv[64];
          tmem_ld64_issue(scol, sv);
          tmem_ld64_wait(sv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sfree(b));
          // P for all 64 heads first, then the stores (the running maxima are read without a
          // store in between)
          uint32_t pw[32];
#pragma unroll
          for (int pc = 0; pc < 8; ++pc) {          // heads 8 pc .. 8 pc + 7
            const float4 m0 = reinterpret_cast<const float4*>(mrun)[2 * pc];
            const float4 m1 = reinterpret_cast<const float4*>(mrun)[2 * pc + 1];
            const float mm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int h = 8 * pc + 2 * e;
              const float p0 = live ? ex2(__uint_as_float(sv[h]) * a.scale_log2 - mm[2 * e]) : 0.f;
              const float p1 = live ? ex2(__uint_as_float(sv[h + 1]) * a.scale_log2 - mm[2 * e + 1]) : 0.f;
              const __nv_bfloat162 pr = __floats2bfloat162_rn(p0, p1);
              pw[4 * pc + e] = *reinterpret_cast<const uint32_t*>(&pr);
            }
          }
          uint8_t* prow = p_s + j * 128;
#pragma unroll
          for (int pc = 0; pc < 8; ++pc)
            *reinterpret_cast<uint4*>(prow + ((pc ^ (j & 7)) << 4)) =
                make_uint4(pw[4 * pc], pw[4 * pc + 1], pw[4 * pc + 2], pw[4 * pc + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        mbar_arrive(pfull);
      }
      ok = group_all(ok);
      // out[t, h, j] = O^T[j, h] / (L[h] + 2^(sink - m))
      if (ok) ok = mbar_wait(pfree, (uint32_t)(ntiles - 1) & 1u, limit, abort_flag);
      ok = group_all(ok);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {          // heads 32 hh .. 32 hh + 31
          uint32_t o[32], l[32];
          tmem_ld32(tl + kColO + 32u * (uint32_t)hh, o);
          tmem_ld32(tl + kColL + 32u * (uint32_t)hh, l);
          if (S == 1) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int h = 32 * hh + e;
              const float den = __uint_as_float(l[e]) + ex2(sink2[h] - mrun[h]);
              orow[h * kDim + j] = den > 0.f ? __uint_as_float(o[e]) / den : 0.f;
            }
          } else {                                // unnormalised, relative to mrun; the sink is added once
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              opart[(32 * hh + e) * kDim + j] = __uint_as_float(o[e]);
              if (j == 32 * hh + e) lpart[j] = __uint_as_float(l[e]);
            }
          }
        }
      } else {
        if (gt == 0) raise_error(DSA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (S > 1) {
    // every CTA of the row's cluster holds its partial (O, L, running max); CTA r combines
    // heads [r * 64 / S, (r + 1) * 64 / S) from all of them:
    //   out = sum_p 2^(m_p - M) O_p / (sum_p 2^(m_p - M) L_p + 2^(sink - M)), M = max(sink, m_p).
    // Every thread of every CTA passes both cluster barriers exactly once (the second one
    // keeps each CTA's shared memory alive until its peers have read it).
    cluster_sync_all();
    if (warp > 0) {
      const int j = 32 * (warp & 3) + lane;
      const int hs = kHeads / S;
      float* orow = a.out + t * (kHeads * kDim);
      for (int h = rank * hs; h < (rank + 1) * hs; ++h) {
        float M = sink2[h];
        for (int r = 0; r < S; ++r) M = fmaxf(M, ld_peer(mrun + h, (uint32_t)r));
        float num = 0.f, den = 0.f;
        if (M > -INFINITY) {
          den = ex2(sink2[h] - M);
          for (int r = 0; r < S; ++r) {
            const float f = ex2(ld_peer(mrun + h, (uint32_t)r) - M);
            num += f * ld_peer(reinterpret_cast<const float*>(x_s) + h * kDim + j, (uint32_t)r);
            den += f * ld_peer(red + h, (uint32_t)r);
          }
        }
        orow[h * kDim + j] = den > 0.f ? num / den : 0.f;
      }
    }
    cluster_sync_all();
  }
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_sparse_attn(const uint16_t* q, int64_t T, const int32_t* sel, int k, const uint8_t* fp4,
                               const uint8_t* scale, int64_t num_blocks, int bs, const int32_t* table,
                               int64_t bt_stride, int next_n, const float* sink, float softmax_scale, float* out,
                               int num_sms, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const size_t smem = attn_smem_bytes(k);
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // A batch too small to fill the GPU (two CTAs per SM) splits each row's selection over a
  // cluster of 2 or 4 CTAs (at most one per tile), combined through distributed shared memory.
  const int nall = (k + kTile - 1) / kTile;
  int split = 1;
  while (split < 4 && (int64_t)T * split * 2 <= (int64_t)2 * num_sms && 2 * split <= nall) split *= 2;
  AttnArgs a{q, sel, k, fp4, scale, num_blocks, bs, table, bt_stride, next_n, sink,
             (float)((double)softmax_scale * 1.4426950408889634), out, split};
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(T * split));
  cfg.blockDim = dim3(32 + kGroup);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)split;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, sparse_attn_kernel, a);
  note_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

size_t sparse_attn_smem_bytes(int k) { return attn_smem_bytes(k); }
int sparse_attn_max_topk() { return kMaxTopk; }

DSA_DEFINE_TU_ERROR_ACCESSORS(attn)

}  // namespace dsa
