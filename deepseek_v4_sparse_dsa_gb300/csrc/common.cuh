// Device-side building blocks shared by the kernels of this library (sm_103a).
//
//  * per-translation-unit error word and wait limit (see dsa.h, dsa_device_error);
//  * bounded mbarrier waits (time limit read from %globaltimer, never a hang);
//  * TMA (cp.async.bulk.tensor) and tcgen05 (MMA into tensor memory) wrappers;
//  * the ranking key of the top-k tie rule and a shared-memory top-k engine (candidate
//    buffer, histogram cut-back, radix select, prefix-sum compaction, bitonic sorts in
//    shared memory or in one warp's registers) used by the fused indexer, the standalone
//    top-k and the merge of partial top-k lists;
//  * the layout of the fused call's work plan and programmatic-dependent-launch hooks.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

// ---------------------------------------------------------------------------------
// Error word and wait limit.  Each translation unit has its own copy (no relocatable
// device code); the host reads and clears all of them in dsa_device_error.
// ---------------------------------------------------------------------------------
static __device__ unsigned int g_error_word;
static __device__ unsigned long long g_wait_limit_ns;

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;   // 2 s
constexpr unsigned long long kCleanupWaitNs = 2000000000ull;   // waits for own copies on abort

__device__ __forceinline__ void raise_error(unsigned int bits) { atomicOr(&g_error_word, bits); }

__device__ __forceinline__ unsigned long long wait_limit_ns() {
  unsigned long long v = *(volatile unsigned long long*)&g_wait_limit_ns;
  return v == 0 ? kDefaultWaitNs : v;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------------
// Shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Gives up after
// `limit_ns` (or as soon as *abort becomes non-zero) and returns false; the caller
// then abandons its work.  Never spins forever.  (try_wait itself may suspend the
// thread for a while before it reports an incomplete phase, so the clock and the
// abort flag are read after every failed attempt.)
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns,
                                          const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of the box at (x = inner element, y = row) into shared memory,
// completing `bytes` of transaction count on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from global
// to shared memory, completing that many bytes of transaction count on the mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// ---------------------------------------------------------------------------------
// Work plan of the fused score + top-k (written by plan_kernel, read by the indexer and
// merge kernels).  Query groups lie end to end on a line; group u spans positions
// [a0, a1): `cost` positions for its fixed per-item cost, then one per key tile.  The
// line is cut into slices of Q positions, one per CTA.  A group whose tiles fall in more
// than one slice is split: each of those slices ranks its piece into an unsorted top-k
// list in slot 2 * slice (the piece starts at the slice start: the "head") or
// 2 * slice + 1 (the piece ends the slice: the "tail"); a slice has at most one of each.
// ---------------------------------------------------------------------------------
// Header (int32): Q, line length, split-group count, cost, mode, work counter, 0, 0.
// Mode kPlanSlices: CTA i takes slice i.  Mode kPlanGroups (every group is short next
// to a slice): CTAs take whole groups from a longest-first list through the counter.
constexpr int kPlanHeader = 8;
constexpr int kPlanSlices = 0;
constexpr int kPlanGroups = 1;

__device__ __forceinline__ int first_tile_slice(int a0, int cost, int Q) { return (a0 + cost) / Q; }
__device__ __forceinline__ int last_tile_slice(int a1, int Q) { return (a1 - 1) / Q; }

__device__ __forceinline__ bool group_is_split(int a0, int a1, int cost, int Q) {
  return a1 - a0 > cost && first_tile_slice(a0, cost, Q) != last_tile_slice(a1, Q);
}

__device__ __forceinline__ int split_slot(int slice, int a0, int cost, int Q) {
  return 2 * slice + ((a0 + cost > slice * Q) ? 1 : 0);
}

// ---------------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with the programmatic-serialisation
// attribute may start while the kernel before it in the stream is still running; it
// must call grid_dependency_wait() before touching anything that kernel writes (the
// wait returns once that kernel has completed and its writes are visible; without the
// attribute it returns at once).  grid_launch_dependents() lets the next such kernel
// start early.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the 128-byte
// swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms packed back to back.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);          // start address
  d |= (uint64_t)(16u >> 4) << 16;                 // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptors: fp32 accumulate, both operands K-major, M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_e4m3(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled contraction (kind::mxf8f6f4, one E8M0 scale per 32 elements along K of
// each operand row; fp32 accumulate; both operands K-major): A holds E2M1 codes in the
// padded shared layout (16 codes = 8 packed bytes followed by 8 unused bytes, so a row of
// 128 codes spans 128 bytes like an E4M3 row), B holds E4M3 codes.  The scale bytes are
// read from tensor memory: byte `a_sf` (`b_sf`) of the 32-bit cells at the given columns
// serves the 32 elements of this K step.  For M = 128 the scales of operand row
// r = l + 32 j sit in column j of lane l, the same in each of the four lane quarters
// (measured: a layout with row r in lane r scores only the first 32 rows right).
__host__ __device__ constexpr uint32_t idesc_mx_e2m1_e4m3(int M, int N, uint32_t a_sf, uint32_t b_sf) {
  return (b_sf << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | (a_sf << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t tmem_sfa,
                                       uint32_t tmem_sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(tmem_sfa), "r"(tmem_sfb), "r"(accumulate)
      : "memory");
}

// Each thread of the warp writes 4 consecutive 32-bit columns of its own TMEM lane (the
// warp's lane quarter is given in taddr); tmem_st_wait completes the warp's stores.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Arrive on an mbarrier once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Each thread of the warp reads 64 consecutive 32-bit columns of its own TMEM lane, in
// two steps so the load of one block of columns can overlap work on the previous one:
// tmem_ld64_issue starts the load, tmem_ld64_wait completes every load the thread has
// issued and marks `r` as written only then (its registers are operands, so the compiler
// cannot move their uses above the wait).
__device__ __forceinline__ void tmem_ld64_issue(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld64_wait(uint32_t (&r)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63]) : : "memory");
}

// ---------------------------------------------------------------------------------
// Ranking key of the tie rule: larger value first, then smaller index.
// High 32 bits: order-preserving image of the fp32 value (-0.0 folded onto +0.0);
// low 32 bits: ~index.  Distinct indices give distinct keys; every real candidate
// has a key > 0, so 0 marks an empty slot.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ float canon_zero(float v) {
  return __float_as_uint(v) == 0x80000000u ? 0.0f : v;
}

__device__ __forceinline__ uint32_t ord_f32(float v) {
  uint32_t u = __float_as_uint(canon_zero(v));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float f32_of_ord(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t rank_key(float v, uint32_t j) {
  return ((uint64_t)ord_f32(v) << 32) | (uint64_t)(~j);
}

__device__ __forceinline__ int32_t index_of_key(uint64_t key) { return (int32_t)(~(uint32_t)key); }
__device__ __forceinline__ float value_of_key(uint64_t key) { return f32_of_ord((uint32_t)(key >> 32)); }

// -inf and NaN are never candidates.
__device__ __forceinline__ bool is_candidate(float v) { return v > -INFINITY; }

// ---------------------------------------------------------------------------------
// Shared-memory top-k engine.  Run by a group of NT threads (a multiple of 128) that
// synchronise on named barrier `bar` (1 unless given); `tid` = 0..NT-1 within the group.
// ---------------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ void group_sync(int bar = 1) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(NT) : "memory");
}

struct EngineScratch {
  uint32_t hist[256];
  uint32_t pick[4];
};

// Appends `key` to buf[*cnt] when `take` is set; warp-aggregated atomics.  All 32
// lanes of the warp must call it together.  A slot at or past `cap` is never written:
// the key is dropped and DSA_DEVERR_OVERFLOW raised, with the call site (1..255) in bits
// 8..15 of the error word (the callers size their buffers so that this cannot happen;
// the check keeps a broken invariant from touching memory it does not own).
__device__ __forceinline__ void engine_append(uint64_t* buf, uint32_t* cnt, uint64_t key, bool take,
                                              uint32_t cap, uint32_t site) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t m = __ballot_sync(0xFFFFFFFFu, take);
  if (m == 0) return;
  uint32_t base = 0;
  const uint32_t leader = __ffs(m) - 1;
  if (lane == leader) base = atomicAdd(cnt, (uint32_t)__popc(m));
  base = __shfl_sync(0xFFFFFFFFu, base, leader);
  if (take) {
    const uint32_t slot = base + __popc(m & ((1u << lane) - 1u));
    if (slot < cap) buf[slot] = key;
    else raise_error(DSA_DEVERR_OVERFLOW | ((site & 0xFFu) << 8));
  }
}

// engine_append for NQ candidate buffers at once (buffer q at buf + q * stride, count
// cnt[q]): one round of shared atomics, issued back to back by lane 0, for all of them.
template <int NQ>
__device__ __forceinline__ void engine_append_multi(uint64_t* buf, size_t stride, uint32_t* cnt,
                                                    const uint64_t (&key)[NQ], const bool (&take)[NQ],
                                                    uint32_t cap, uint32_t site) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t below = (1u << lane) - 1u;
  uint32_t m[NQ], base[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    m[q] = __ballot_sync(0xFFFFFFFFu, take[q]);
    base[q] = 0u;
  }
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (m[q]) base[q] = atomicAdd(&cnt[q], (uint32_t)__popc(m[q]));
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (m[q] == 0u) continue;
    const uint32_t b = __shfl_sync(0xFFFFFFFFu, base[q], 0);
    if (take[q]) {
      const uint32_t slot = b + __popc(m[q] & below);
      if (slot < cap) buf[q * stride + slot] = key[q];
      else raise_error(DSA_DEVERR_OVERFLOW | ((site & 0xFFu) << 8));
    }
  }
}

// hist[bin] += 1 for every lane with `take`: one shared atomic per lane (measured
// faster on sm_103 than aggregating equal bins with a match first, even when the keys
// of a candidate set crowd into a few bins).  All 32 lanes must call it together.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool take, uint32_t bin) {
  if (take) atomicAdd(&hist[bin], 1u);
}

// Picks the digit of the current radix pass: the bin holding the `need`-th largest key,
// scanning hist from the top.  Run by warp 0 of the group; results in sc->pick.
__device__ __forceinline__ void pick_digit(uint32_t* hist, uint32_t* pick, uint32_t need, int tid) {
  uint32_t c[8], sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = hist[255 - 8 * tid - i];
    sum += c[i];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (tid >= o) incl += y;
  }
  const uint32_t excl = incl - sum;
  if (tid == 31) pick[3] = incl;    // total count of this pass
  if (tid == 31 && need > incl) pick[0] = 0xFFFFFFFFu;   // no such bin: inconsistent input
  if (excl < need && need <= incl) {
    uint32_t above = excl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (above < need && need <= above + c[i]) {
        pick[0] = 255u - 8u * tid - i;
        pick[1] = above;
        pick[2] = c[i];
      }
      above += c[i];
    }
  }
}

// Smallest key T such that exactly k of the distinct nonzero keys in buf[0, n) are >= T
// (the k-th largest key, or a lower bound of it sharing all bits that decide the set);
// 1 when there are at most k of them.  Most-significant-digit-first radix select over
// 8-bit digits, starting at the highest byte in which the keys differ (one AND / OR
// reduction finds it: candidates share their sign and exponent bits, and a pass over a
// digit they all share would only pile every key into one bin); zero slots are ignored.
template <int NT>
__device__ uint64_t engine_select(const uint64_t* buf, int n, int k, EngineScratch* sc, int tid, int bar = 1) {
  constexpr int NW = NT / 32;
  static_assert(5 * NW <= 256, "group size");
  const int lane = tid & 31, w = tid >> 5;
  uint64_t kand = ~0ull, kor = 0ull;
  uint32_t nz = 0;
  for (int e = tid; e < n; e += NT) {
    const uint64_t key = buf[e];
    if (key) {
      kand &= key;
      kor |= key;
      ++nz;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    kand &= __shfl_xor_sync(0xFFFFFFFFu, kand, o);
    kor |= __shfl_xor_sync(0xFFFFFFFFu, kor, o);
    nz += __shfl_xor_sync(0xFFFFFFFFu, nz, o);
  }
  uint32_t* red = sc->hist;                         // per warp: and (2 words), or (2 words), count
  if (lane == 0) {
    red[5 * w + 0] = (uint32_t)kand;
    red[5 * w + 1] = (uint32_t)(kand >> 32);
    red[5 * w + 2] = (uint32_t)kor;
    red[5 * w + 3] = (uint32_t)(kor >> 32);
    red[5 * w + 4] = nz;
  }
  group_sync<NT>(bar);
  kand = ~0ull;
  kor = 0ull;
  nz = 0;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    kand &= (uint64_t)red[5 * i] | ((uint64_t)red[5 * i + 1] << 32);
    kor |= (uint64_t)red[5 * i + 2] | ((uint64_t)red[5 * i + 3] << 32);
    nz += red[5 * i + 4];
  }
  group_sync<NT>(bar);                              // red is read before hist reuses it
  if (nz <= (uint32_t)k) return 1ull;               // at most k keys: take them all
  const int top = 63 - __clzll(kand ^ kor);         // highest bit in which keys differ
  const int first = top & ~7;                       // its digit
  uint64_t mask = first >= 56 ? 0ull : ~((1ull << (first + 8)) - 1ull);
  uint64_t prefix = kand & mask;
  uint32_t need = (uint32_t)k;
  for (int shift = first; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) sc->hist[i] = 0;
    group_sync<NT>(bar);
    for (int base = 0; base < n; base += NT) {
      const int e = base + tid;
      const uint64_t key = e < n ? buf[e] : 0ull;
      hist_add(sc->hist, key != 0ull && (key & mask) == prefix, (uint32_t)(key >> shift) & 255u);
    }
    group_sync<NT>(bar);
    if (tid < 32) pick_digit(sc->hist, sc->pick, need, tid);   // lane l: digits 255-8l .. 248-8l
    group_sync<NT>(bar);
    const uint32_t d = sc->pick[0], above = sc->pick[1], inbin = sc->pick[2];
    if (d > 255u) {                // counts did not add up: keep everything (never drops a key)
      if (tid == 0) raise_error(DSA_DEVERR_OVERFLOW | (42u << 8));
      group_sync<NT>(bar);
      return 1ull;
    }
    need -= above;
    prefix |= (uint64_t)d << shift;
    mask |= (uint64_t)0xFF << shift;
    if (inbin == need) break;      // every key with this prefix belongs to the set
  }
  group_sync<NT>(bar);             // everyone has read pick[] before it is reused
  return prefix;
}

// Histogram bin of value image o for a cut-back over [lo, lo + span): (o - lo) * mul / 2^32
// with mul = floor(2^32 * kCutBins / span), monotone in o and below kCutBins.
__device__ __forceinline__ uint32_t cut_bin(uint32_t o, uint32_t lo, uint32_t mul) {
  return (uint32_t)(((uint64_t)(o - lo) * mul) >> 32);
}

// Writes the keys of keep[] that are nonzero and >= thr (kByBin: whose cut_bin is at
// least bmin) to the front of buf, in thread order, with one prefix sum over the group
// instead of an atomic per key; *cnt becomes their number; returns the smallest value
// image written.  Every key of buf must already sit in some thread's keep[] (the writes
// may overwrite any slot).  Uses sc->hist[0, 2 * NT/32) as scratch; ends with a group
// barrier.
template <int NT, int MAXPER, bool kByBin>
__device__ __forceinline__ uint32_t engine_scatter(uint64_t* buf, uint32_t* cnt, const uint64_t (&keep)[MAXPER],
                                                   uint64_t thr, uint32_t lo, uint32_t mul, uint32_t bmin,
                                                   EngineScratch* sc, int tid, int bar) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, w = tid >> 5;
  uint32_t mine = 0, omin = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < MAXPER; ++i) {
    const uint32_t o = (uint32_t)(keep[i] >> 32);
    const bool t = kByBin ? (keep[i] != 0ull && cut_bin(o, lo, mul) >= bmin) : (keep[i] != 0ull && keep[i] >= thr);
    mine += t ? 1u : 0u;
    if (t) omin = min(omin, o);
  }
  for (int o = 16; o > 0; o >>= 1) omin = min(omin, __shfl_xor_sync(0xFFFFFFFFu, omin, o));
  if (lane == 0) sc->hist[NW + w] = omin;
  uint32_t incl = mine;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc->hist[w] = incl;
  group_sync<NT>(bar);
  uint32_t off = incl - mine, total = 0;
  omin = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const uint32_t c = sc->hist[i];
    if (i < w) off += c;
    total += c;
    omin = min(omin, sc->hist[NW + i]);
  }
#pragma unroll
  for (int i = 0; i < MAXPER; ++i) {
    const bool t = kByBin ? (keep[i] != 0ull && cut_bin((uint32_t)(keep[i] >> 32), lo, mul) >= bmin)
                          : (keep[i] != 0ull && keep[i] >= thr);
    if (t) buf[off++] = keep[i];
  }
  if (tid == 0) *cnt = total;
  group_sync<NT>(bar);
  return omin;
}

// Cheap cut-back of a candidate buffer that only has to stay a superset of its top-k:
// one 512-bin histogram of the keys' values (bins linear in the order-preserving image
// of the value, between its smallest and largest) gives the bin holding the k-th key;
// the keys in that bin and above are kept, packed to the front (*cnt = their number),
// at least k of them, and the function returns T = (smallest kept value image) << 32,
// a threshold at or below the k-th key.  Returns 0 and leaves buf alone when
// the histogram cannot bring the count to `room` or less (values too concentrated, e.g.
// ties) or there are at most k keys; the caller then selects exactly.  `bins` holds 512
// words of shared scratch; needs n <= NT * MAXPER.
constexpr int kCutBins = 512;

template <int NT, int MAXPER>
__device__ uint64_t engine_cut_approx(uint64_t* buf, uint32_t* cnt, int n, int k, uint32_t room, uint32_t* bins,
                                      EngineScratch* sc, int tid, int bar = 1) {
  constexpr int NW = NT / 32;
  constexpr int BPT = kCutBins / NT;               // bins per thread in the scan
  static_assert(kCutBins % NT == 0 && NW <= 16, "group size");
  const int lane = tid & 31, w = tid >> 5;
  uint64_t keep[MAXPER];
  uint32_t lo = 0xFFFFFFFFu, hi = 0u, nz = 0u;
#pragma unroll
  for (int i = 0; i < MAXPER; ++i) {
    const int e = tid + i * NT;
    keep[i] = (e < n) ? buf[e] : 0ull;
    if (keep[i]) {
      const uint32_t o = (uint32_t)(keep[i] >> 32);
      lo = min(lo, o);
      hi = max(hi, o);
      ++nz;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
    nz += __shfl_xor_sync(0xFFFFFFFFu, nz, o);
  }
  uint32_t* wred = sc->hist;                        // [0, 3 * NW): per-warp lo, hi, count
  if (lane == 0) {
    wred[w] = lo;
    wred[NW + w] = hi;
    wred[2 * NW + w] = nz;
  }
  for (int i = tid; i < kCutBins; i += NT) bins[i] = 0u;
  group_sync<NT>(bar);
  lo = 0xFFFFFFFFu;
  hi = 0u;
  nz = 0u;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    lo = min(lo, wred[i]);
    hi = max(hi, wred[NW + i]);
    nz += wred[2 * NW + i];
  }
  if (nz <= (uint32_t)k || hi == lo) {
    group_sync<NT>(bar);                               // wred is read before it is reused
    return 0ull;
  }
  const uint64_t span = (uint64_t)(hi - lo) + 1u;
  const uint32_t mul = (uint32_t)min(((uint64_t)kCutBins << 32) / span, (uint64_t)0xFFFFFFFFu);
#pragma unroll
  for (int i = 0; i < MAXPER; ++i)
    if (keep[i]) atomicAdd(&bins[cut_bin((uint32_t)(keep[i] >> 32), lo, mul)], 1u);
  group_sync<NT>(bar);
  // bin b* holding the k-th key from the top: thread tid scans bins
  // [kCutBins - (tid + 1) * BPT, kCutBins - tid * BPT) top down
  uint32_t c[BPT], sum = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    c[i] = bins[kCutBins - 1 - tid * BPT - i];
    sum += c[i];
  }
  uint32_t incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t* wsum = sc->hist + 3 * NW;               // [3 * NW, 4 * NW): per-warp totals
  if (lane == 31) wsum[w] = incl;
  group_sync<NT>(bar);
  uint32_t before = 0;
  for (int i = 0; i < w; ++i) before += wsum[i];
  uint32_t above = before + incl - sum;
  if (above < (uint32_t)k && (uint32_t)k <= above + sum) {
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (above < (uint32_t)k && (uint32_t)k <= above + c[i]) {
        sc->pick[0] = (uint32_t)(kCutBins - 1 - tid * BPT - i);
        sc->pick[1] = above + c[i];
      }
      above += c[i];
    }
  }
  group_sync<NT>(bar);
  const uint32_t b = sc->pick[0], count = sc->pick[1];
  if (count > room) {
    group_sync<NT>(bar);
    return 0ull;
  }
  // keys in bins >= b stay; the threshold is the smallest value image among them
  const uint32_t tord = engine_scatter<NT, MAXPER, true>(buf, cnt, keep, 0ull, lo, mul, b, sc, tid, bar);
  return (uint64_t)tord << 32;
}

// Exact cut-back of a candidate set held in registers: keep[] holds every candidate of
// the set (distinct nonzero keys; zero = empty) spread over the group's threads.  The k
// largest (all of them when there are at most k) are written to the front of buf, *cnt
// becomes their number, and the k-th largest key (1 when all are kept) is returned: the
// set's new threshold.  One 512-bin histogram of the value images finds the bin holding
// the k-th key; the few keys in that bin are sorted by one warp to name the k-th key
// exactly; only when the bin holds more than 64 keys (values packed closely, e.g. ties)
// does the exact radix select over the (compacted) set decide.  `bins` holds 512 words of
// shared scratch and must be 8-byte aligned (its front is reused as a list of 64-bit
// keys); buf must have room for every candidate (the writes may overwrite any of the
// slots the candidates came from: they are all in keep[] already).
template <int KPL>
__device__ __forceinline__ void warp_sort_regs(uint64_t (&x)[KPL]);

template <int NT, int MAXPER>
__device__ uint64_t engine_cut_exact_keep(uint64_t* buf, uint32_t* cnt, const uint64_t (&keep)[MAXPER], int k,
                                          uint32_t* bins, EngineScratch* sc, int tid, int bar = 1) {
  constexpr int NW = NT / 32;
  constexpr int BPT = kCutBins / NT;
  static_assert(kCutBins % NT == 0 && NW <= 16, "group size");
  const int lane = tid & 31, w = tid >> 5;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u, nz = 0u;
#pragma unroll
  for (int i = 0; i < MAXPER; ++i) {
    if (keep[i]) {
      const uint32_t o = (uint32_t)(keep[i] >> 32);
      lo = min(lo, o);
      hi = max(hi, o);
      ++nz;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
    nz += __shfl_xor_sync(0xFFFFFFFFu, nz, o);
  }
  uint32_t* wred = sc->hist;                        // [0, 3 * NW): per-warp lo, hi, count
  if (lane == 0) {
    wred[w] = lo;
    wred[NW + w] = hi;
    wred[2 * NW + w] = nz;
  }
  for (int i = tid; i < kCutBins; i += NT) bins[i] = 0u;
  group_sync<NT>(bar);
  lo = 0xFFFFFFFFu;
  hi = 0u;
  nz = 0u;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    lo = min(lo, wred[i]);
    hi = max(hi, wred[NW + i]);
    nz += wred[2 * NW + i];
  }
  group_sync<NT>(bar);                              // wred is read before it is reused
  if (nz <= (uint32_t)k) {                          // keep them all, compacted
    engine_scatter<NT, MAXPER, false>(buf, cnt, keep, 1ull, 0u, 0u, 0u, sc, tid, bar);
    return 1ull;
  }
  const uint64_t span = (uint64_t)(hi - lo) + 1u;
  const uint32_t mul = (uint32_t)min(((uint64_t)kCutBins << 32) / span, (uint64_t)0xFFFFFFFFu);
#pragma unroll
  for (int i = 0; i < MAXPER; ++i)
    if (keep[i]) atomicAdd(&bins[cut_bin((uint32_t)(keep[i] >> 32), lo, mul)], 1u);
  group_sync<NT>(bar);
  // bin b holding the k-th key from the top, and the count of keys in the bins above it
  uint32_t c[BPT], sum = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    c[i] = bins[kCutBins - 1 - tid * BPT - i];
    sum += c[i];
  }
  uint32_t incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t* wsum = sc->hist + 3 * NW;               // [3 * NW, 4 * NW): per-warp totals
  if (lane == 31) wsum[w] = incl;
  group_sync<NT>(bar);
  uint32_t before = 0;
  for (int i = 0; i < w; ++i) before += wsum[i];
  uint32_t above = before + incl - sum;
  if (above < (uint32_t)k && (uint32_t)k <= above + sum) {
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (above < (uint32_t)k && (uint32_t)k <= above + c[i]) {
        sc->pick[0] = (uint32_t)(kCutBins - 1 - tid * BPT - i);
        sc->pick[1] = above;                        // keys in the bins above b
        sc->pick[2] = c[i];                         // keys in bin b
      }
      above += c[i];
    }
  }
  group_sync<NT>(bar);
  const uint32_t b = sc->pick[0], abv = sc->pick[1], inb = sc->pick[2];
  uint64_t thr;
  if (inb <= 64u) {
    // the keys of bin b into a short list (bins is free again), sorted by warp 0
    uint64_t* list = reinterpret_cast<uint64_t*>(bins);
    if (tid == 0) sc->pick[3] = 0u;
    if (tid < 64) list[tid] = 0ull;
    group_sync<NT>(bar);
#pragma unroll
    for (int i = 0; i < MAXPER; ++i) {
      if (keep[i] && cut_bin((uint32_t)(keep[i] >> 32), lo, mul) == b) {
        const uint32_t at = atomicAdd(&sc->pick[3], 1u);
        if (at < 64u) list[at] = keep[i];
      }
    }
    group_sync<NT>(bar);
    if (w == 0) {
      uint64_t x[2] = {list[lane], list[32 + lane]};
      warp_sort_regs<2>(x);                         // descending: element e = r * 32 + lane
      const uint32_t e = (uint32_t)k - abv - 1u;    // the (k - abv)-th largest of the bin
      if (lane == (int)(e & 31u)) list[64] = x[e >> 5];
    }
    group_sync<NT>(bar);
    thr = list[64];
  } else {
    // compact the set to the front of buf, then the exact radix select over it
    engine_scatter<NT, MAXPER, false>(buf, cnt, keep, 1ull, 0u, 0u, 0u, sc, tid, bar);
    thr = engine_select<NT>(buf, (int)nz, k, sc, tid, bar);
  }
  engine_scatter<NT, MAXPER, false>(buf, cnt, keep, thr, 0u, 0u, 0u, sc, tid, bar);
  return thr;
}

// Keeps the keys >= thr of buf[0, n), packed to the front; *cnt becomes their
// number.  Holds the keys in registers meanwhile: needs n <= NT * MAXPER.  The caller
// has passed a group barrier since buf and n were last written.
template <int NT, int MAXPER>
__device__ void engine_compact(uint64_t* buf, uint32_t* cnt, int n, uint64_t thr, EngineScratch* sc, int tid,
                               int bar = 1) {
  uint64_t keep[MAXPER];
#pragma unroll
  for (int i = 0; i < MAXPER; ++i) {
    const int e = tid + i * NT;
    keep[i] = (e < n) ? buf[e] : 0ull;
  }
  engine_scatter<NT, MAXPER, false>(buf, cnt, keep, thr, 0u, 0u, 0u, sc, tid, bar);
}

// The top k of a candidate set cand[0, n) (distinct nonzero keys; zero slots ignored), in
// rank order, by value bins: the candidates are binned by value image (kCutBins linear bins
// over their range, as in a cut-back); one scan from the top finds the bin b* that holds the
// k-th largest (the lowest bin when there are fewer than k); the candidates of the bins at
// or above b* are gathered in bin order, and each ranks as the count in the bins above its
// own plus the larger keys of its own bin.  Key r goes to row_idx[r] / row_val[r] (nothing
// is written when row_idx is null); *m_out = min(k, candidates).  Returns false, having
// written nothing, when bin b* holds more than max_bin candidates (values crowded together):
// the caller then selects exactly.  Scratch: tmp (k + max_bin slots), start and bins
// (kCutBins words each), red (2 * NT / 32 words), pick (2 words).  Equal keys (possible only
// in stale lists) raise DSA_DEVERR_OVERFLOW.
template <int NT>
__device__ bool engine_topk_binned(const uint64_t* cand, int n, int k, uint64_t* tmp, uint32_t max_bin,
                                   uint32_t* start, uint32_t* bins, uint32_t* red, uint32_t* pick, int tid,
                                   int32_t* row_idx, float* row_val, int* m_out, int bar = 1) {
  constexpr int NW = NT / 32;
  constexpr int BPT = kCutBins / NT;               // bins per thread in the scan
  static_assert(kCutBins % NT == 0 && NW <= 16, "group size");
  const int lane = tid & 31, w = tid >> 5;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int e = tid; e < n; e += NT) {
    const uint64_t key = cand[e];
    if (key) {
      lo = min(lo, (uint32_t)(key >> 32));
      hi = max(hi, (uint32_t)(key >> 32));
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
  }
  if (lane == 0) {
    red[w] = lo;
    red[NW + w] = hi;
  }
  for (int i = tid; i < kCutBins; i += NT) bins[i] = 0u;
  group_sync<NT>(bar);
  lo = 0xFFFFFFFFu;
  hi = 0u;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    lo = min(lo, red[i]);
    hi = max(hi, red[NW + i]);
  }
  const uint64_t span = hi >= lo ? (uint64_t)(hi - lo) + 1u : 1u;
  const uint32_t mul = (uint32_t)min(((uint64_t)kCutBins << 32) / span, (uint64_t)0xFFFFFFFFu);
  for (int e = tid; e < n; e += NT) {
    const uint64_t key = cand[e];
    if (key) atomicAdd(&bins[cut_bin((uint32_t)(key >> 32), lo, mul)], 1u);
  }
  group_sync<NT>(bar);
  // start[b]: the candidates in the bins above b; thread tid scans bins
  // kCutBins - 1 - tid * BPT - i, i < BPT (top down)
  uint32_t c[BPT], sum = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    c[i] = bins[kCutBins - 1 - tid * BPT - i];
    sum += c[i];
  }
  uint32_t incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  group_sync<NT>(bar);                             // red is rewritten
  if (lane == 31) red[w] = incl;
  group_sync<NT>(bar);
  uint32_t st = incl - sum;
  for (int i = 0; i < w; ++i) st += red[i];
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    const int b = kCutBins - 1 - tid * BPT - i;
    start[b] = st;
    bins[b] = st;                                  // running slot of the gather
    if (st < (uint32_t)k && (uint32_t)k <= st + c[i]) {   // b* (one bin at most)
      pick[0] = (uint32_t)b;
      pick[1] = st + c[i];
    }
    if (b == 0 && st + c[i] < (uint32_t)k) {      // fewer than k candidates: every bin
      pick[0] = 0u;
      pick[1] = st + c[i];
    }
    st += c[i];
  }
  group_sync<NT>(bar);
  const uint32_t bstar = pick[0], total = pick[1];   // total: the candidates in bins >= b*
  const bool crowded = total - start[bstar] > max_bin;
  group_sync<NT>(bar);                             // pick and start read before any reuse
  if (crowded) return false;
  for (int e = tid; e < n; e += NT) {
    const uint64_t key = cand[e];
    if (!key) continue;
    const uint32_t kb = cut_bin((uint32_t)(key >> 32), lo, mul);
    if (kb >= bstar) tmp[atomicAdd(&bins[kb], 1u)] = key;
  }
  group_sync<NT>(bar);
  for (uint32_t q = (uint32_t)tid; q < total; q += NT) {
    const uint64_t key = tmp[q];
    const uint32_t kb = cut_bin((uint32_t)(key >> 32), lo, mul);
    const uint32_t s1 = bins[kb];
    uint32_t r = start[kb], eq = 0;
    for (uint32_t j = start[kb]; j < s1; ++j) {
      const uint64_t x = tmp[j];
      r += x > key ? 1u : 0u;
      eq += x == key ? 1u : 0u;
    }
    if (eq > 1) raise_error(DSA_DEVERR_OVERFLOW | (33u << 8));
    if (r < (uint32_t)k && row_idx != nullptr) {
      row_idx[r] = index_of_key(key);
      if (row_val) row_val[r] = value_of_key(key);
    }
  }
  *m_out = (int)min(total, (uint32_t)k);
  group_sync<NT>(bar);                             // tmp, start and bins free again
  return true;
}

// Copies the keys >= thr of src[0, n) to the front of dst (capacity dcap); *cnt becomes
// their number.
template <int NT>
__device__ void engine_compact_to(const uint64_t* src, uint64_t* dst, uint32_t* cnt, int n, uint64_t thr,
                                  int tid, uint32_t dcap) {
  if (tid == 0) *cnt = 0;
  group_sync<NT>();
  for (int base = 0; base < n; base += NT) {
    const int e = base + tid;
    const uint64_t key = e < n ? src[e] : 0ull;
    engine_append(dst, cnt, key, key != 0ull && key >= thr, dcap, 2u);
  }
  group_sync<NT>();
}

// Sorts nlist lists in place, each of P (power of two) keys at buf + l * stride,
// in descending key order (rank order).  Slots past a list's count must hold 0.
template <int NT>
__device__ void engine_sort(uint64_t* buf, int stride, int nlist, int P, int tid) {
  const int pairs = P >> 1;
  for (int size = 2; size <= P; size <<= 1) {
    for (int half = size >> 1; half > 0; half >>= 1) {
      for (int t = tid; t < pairs * nlist; t += NT) {
        const int l = t / pairs, u = t - l * pairs;
        const int i = 2 * u - (u & (half - 1));
        const int j = i + half;
        uint64_t* b = buf + (size_t)l * stride;
        const uint64_t x = b[i], y = b[j];
        const bool desc = (i & size) == 0;
        if ((x < y) == desc) {
          b[i] = y;
          b[j] = x;
        }
      }
      group_sync<NT>();
    }
  }
}

// Sorts 32 * KPL keys held by one warp in registers in descending order; element
// e = r * 32 + lane is x[r] of that lane.  Same bitonic network as engine_sort: pairs
// closer than 32 exchange through shuffles, the others within a thread.
template <int KPL>
__device__ __forceinline__ void warp_sort_regs(uint64_t (&x)[KPL]) {
  const int lane = threadIdx.x & 31;
  constexpr int N = 32 * KPL;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int half = size >> 1; half > 0; half >>= 1) {
      if (half >= 32) {
        const int rh = half >> 5;
#pragma unroll
        for (int r = 0; r < KPL; ++r) {
          if ((r & rh) == 0) {
            const bool desc = ((r * 32 + lane) & size) == 0;
            const uint64_t a = x[r], b = x[r + rh];
            const bool sw = (a < b) == desc;
            x[r] = sw ? b : a;
            x[r + rh] = sw ? a : b;
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < KPL; ++r) {
          const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, x[r], half);
          const bool desc = ((r * 32 + lane) & size) == 0;
          const bool keep_max = ((lane & half) == 0) == desc;
          x[r] = keep_max ? (x[r] > o ? x[r] : o) : (x[r] < o ? x[r] : o);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------
// mxfp4 decode (E2M1 nibbles, low nibble first, times an E8M0 group scale 2^(b-127),
// 0xFF -> 0), shared by the gather and the FP4-key score (xkernels issue #28
// "DeepSeek-V4 serving support -- tracking", comment 2 "What it does").
// ---------------------------------------------------------------------------------
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

// Scale bytes outside the fast decode's reach (which covers 2..252 and 0xFF): 0 and 1
// (subnormal results), 253 and 254 (overflowing ones).  (x + 3) mod 256 maps them to 3, 4, 0, 1 and 0xFF to 2.
__device__ __forceinline__ bool e8m0_off_table(uint32_t b) {
  const uint32_t v = (b + 3u) & 0xFFu;
  return v < 5u && v != 2u;
}

// Any of the four scale bytes packed in `w` outside the fast decode's reach.
__device__ __forceinline__ bool e8m0_word_off_table(uint32_t w) {
  bool r = false;
#pragma unroll
  for (int g = 0; g < 4; ++g) r |= e8m0_off_table((w >> (8 * g)) & 0xFFu);
  return r;
}

// Eight elements (nibble bytes of w, low nibble first) times 2^(b-127) as bf16 pairs,
// by byte permutation, with no table in shared memory.  For one scale byte b (2..252, or 0xFF), the bf16 patterns of the 8 magnitudes (code 0 -> 0, code c >= 1
// -> ((b - 1) << 7) + (c << 6), minus 64 for code 1) are split into their low and high
// bytes, 8 of each in two registers; a word's 8 magnitude codes select from them with
// `prmt` (4 selectors per instruction), two more `prmt` interleave low and high bytes into
// bf16 pairs, and the signs are or-ed in.  Shared-memory table reads of random bytes
// conflict across banks; this form is all ALU work.
struct E2M1Bytes {
  uint32_t lo0, lo1, hi0, hi1;   // low / high bytes of the patterns of codes 0-3 and 4-7
};

__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ E2M1Bytes e2m1_bytes(uint32_t b) {
  const uint32_t e = (b - 1u) << 7;
  uint32_t p01 = e << 16;                            // codes 0, 1 (bf16 pairs)
  uint32_t p23 = (e + 128u) | ((e + 192u) << 16);
  uint32_t p45 = (e + 256u) | ((e + 320u) << 16);
  uint32_t p67 = (e + 384u) | ((e + 448u) << 16);
  if (b == 255u) p01 = p23 = p45 = p67 = 0u;         // scale 0: signed zeros only
  E2M1Bytes t;
  t.lo0 = byte_perm(p01, p23, 0x6420u);
  t.hi0 = byte_perm(p01, p23, 0x7531u);
  t.lo1 = byte_perm(p45, p67, 0x6420u);
  t.hi1 = byte_perm(p45, p67, 0x7531u);
  return t;
}

// Eight elements (nibbles of w, low nibble first) as four bf16 pairs, by the tables of
// e2m1_bytes (scale bytes 2..252 or 0xFF; the others take decode8_exact).
__device__ __forceinline__ uint4 decode8_perm(uint32_t w, const E2M1Bytes& t) {
  const uint32_t m = w & 0x77777777u, sg = w & 0x88888888u;
  const uint32_t l0 = byte_perm(t.lo0, t.lo1, m), h0 = byte_perm(t.hi0, t.hi1, m);
  const uint32_t l1 = byte_perm(t.lo0, t.lo1, m >> 16), h1 = byte_perm(t.hi0, t.hi1, m >> 16);
  uint32_t o0 = byte_perm(l0, h0, 0x5140u), o1 = byte_perm(l0, h0, 0x7362u);
  uint32_t o2 = byte_perm(l1, h1, 0x5140u), o3 = byte_perm(l1, h1, 0x7362u);
  o0 |= ((sg << 12) & 0x8000u) | ((sg << 24) & 0x80000000u);   // nibble k's sign (bit 4k + 3)
  o1 |= ((sg << 4) & 0x8000u) | ((sg << 16) & 0x80000000u);    // to bit 15 or 31 of its pair
  o2 |= ((sg >> 4) & 0x8000u) | ((sg << 8) & 0x80000000u);
  o3 |= ((sg >> 12) & 0x8000u) | (sg & 0x80000000u);
  return make_uint4(o0, o1, o2, o3);
}

// Same, for any scale byte, nibble by nibble.
__device__ __forceinline__ uint4 decode8_exact(uint32_t w, uint32_t b) {
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t byte = (w >> (8 * k)) & 0xFFu;
    o[k] = e2m1_bf16_general(byte & 0xFu, (int)b) | (e2m1_bf16_general(byte >> 4, (int)b) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__host__ __device__ constexpr int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace dsa
