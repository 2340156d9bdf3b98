// Device building blocks shared by the kernels of this library (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/w8a8.h"

namespace w8a8 {

// A pipeline wait gives up after this many SM clock cycles (about one second at GB300 clocks) and
// reports W8A8_DEV_WAIT_TIMEOUT instead of spinning forever.  The cycle counter is read once per
// suspended poll (each poll sleeps at most kSuspendHintNs).
constexpr long long kWaitTimeoutCycles = 2000000000ll;

// The bound of the one wait that the W8A8_FLAG_TEST_STALL hook sets up to run out (a few
// milliseconds at GB300 clocks), so that a test of the device fault path ends quickly.
constexpr long long kTestStallCycles = 4000000ll;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier (CTA scope)
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// One non-blocking test of the phase of `parity` (mbarrier.test_wait never waits).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same, but a thread whose phase is not complete stays suspended (issuing nothing) until the
// phase completes or about kSuspendHintNs have passed, instead of returning at once: waiting warps
// then leave the issue slots to the warps that have work.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete.  Bounded: gives up when another thread of the CTA
// has raised *abort, or after `limit` cycles (then records the timeout in *status and raises
// *abort).  Returns true when the phase completed.  The first look is a non-blocking test; after
// that the thread stays suspended in the hinted try_wait until the phase completes (measured on
// GB300: one suspension per blocking wait, resumed about 64 ns after the completing arrival).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, long long limit = kWaitTimeoutCycles) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      atomicOr(status, W8A8_DEV_WAIT_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// Wait for a phase that is sure to complete (copies already issued): bounded by the cycle limit
// only.  Returns false on timeout (recorded in *status).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint32_t* status) {
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity)) return true;
    if (clock64() - t0 > kWaitTimeoutCycles) {
      atomicOr(status, W8A8_DEV_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- thread-block clusters
// Rank of this CTA in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address (shared::cluster window) of the same location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local_smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
  return r;
}

// 16-byte store into another CTA's shared memory (shared::cluster address).
__device__ __forceinline__ void st_cluster_v4f(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

// Cluster-wide barrier: returns once every thread of every CTA in the cluster has arrived; writes
// before it (including into other CTAs' shared memory) are visible after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- bulk copies (TMA engine)
// One-dimensional global -> shared bulk copy completing on `bar` (complete_tx); both addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// The same with an L2 cache policy (used to mark the once-read weight stream evict-first).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- exact int8 -> fp16 pairs
// u holds four int8 values in offset binary (v + 128, v in [-128, 127]).  Each fp16 pattern
// 0x6400 | b is the integer 1024 + b (exponent 2^10, unit spacing), so subtracting 1152 gives v
// exactly.  lo receives bytes (0, 2), hi bytes (1, 3), each as (low half, high half).
__device__ __forceinline__ void offset_bytes_to_half2(uint32_t u, uint32_t& lo, uint32_t& hi) {
  const uint32_t a = (u & 0x00FF00FFu) | 0x64006400u;
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4341);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// ---------------------------------------------------------------- warp MMA
// D += A(16x16 fp16, row) * B(16x8 fp16, col), fp32 accumulate.  Not volatile: the compiler may
// interleave independent MMAs (issue is in order, so a dependent MMA placed right after the one it
// waits for would stall the warp for a full MMA latency).
__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Named barrier among `threads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- split plans (host and device)
// Part i of G equal parts of [0, U): [even_lo(i), even_lo(i + 1)), runs within one of each other.
// 32-bit arithmetic only (i * U < 2^31 at every call site): a 64-bit division is a called
// subroutine on the GPU, and in a kernel prologue its latency delays the first copy.
__host__ __device__ __forceinline__ int even_lo(int i, int U, int G) {
  return (int)((unsigned)(i * U) / (unsigned)G);
}

// Work split of a W8A8 GEMM call: G CTAs share T tiles of KB slabs (U = T * KB slabs, U < 2^31).
//  - Tile-aligned (G >= T): tile t is cut into P_t parts, P_t = c + 1 for the first e tiles and
//    c for the rest (c = G / T, e = G % T), part j of P_t taking slabs [even_lo(j), even_lo(j+1))
//    of the tile's KB.  No CTA crosses a tile, so each CTA finishes exactly one tile segment and
//    P_t CTAs meet in the tile's combine.
//  - Linear (G < T): the tiles are laid end to end and cut into units of 2^qs slabs; CTA i takes
//    a contiguous run of a + 1 (i < r) or a units (a = U' / G, r = U' % G over the U' = U / 2^qs
//    units), which may span several tiles.
// Both cover every slab exactly once with no empty run (G <= U).
struct GemmSplit {
  int T, KB, G;
  int aligned;
  int c, e;   // tile-aligned: parts per tile, tiles with one extra part
  int a, r;   // linear: run length in units, runs one unit longer
  int qs;     // linear: log2 of the slabs per unit (0 or 2)
};

// coarse: the decode kernel's split, whose linear runs go in units of 4 slabs (so every run starts
// on an 8 KiB boundary of the packed weight) when K is a multiple of 128 and the longest run grows
// by at most 3 %.  Measured on GB300 at K = 4096, N = 24576 (96 MiB of weight, 304 CTAs):
// 0.5-1.2 us less per call for M = 1..32 than runs cut at any slab.
inline GemmSplit make_gemm_split(int T, int KB, int G, bool coarse = false) {
  GemmSplit s{};
  s.T = T;
  s.KB = KB;
  s.G = G;
  s.aligned = G >= T;
  s.c = G / T;
  s.e = G % T;
  const int U = T * KB;
  s.qs = 0;
  if (!s.aligned && coarse && KB % 4 == 0 && U / 4 >= G) {
    const long long run1 = (U + G - 1) / G, run4 = 4ll * ((U / 4 + G - 1) / G);
    if (run4 * 100 <= run1 * 103) s.qs = 2;
  }
  s.a = (U >> s.qs) / G;
  s.r = (U >> s.qs) % G;
  return s;
}

// First and one-past-last slab of CTA i.
__host__ __device__ __forceinline__ void gemm_split_run(const GemmSplit& s, int i, int* b0, int* b1) {
  if (s.aligned) {
    const int big = s.e * (s.c + 1);   // CTAs of the tiles cut into c + 1 parts
    int t, j, P;
    if (i < big) {
      P = s.c + 1;
      t = (int)((unsigned)i / (unsigned)P);
      j = i - t * P;
    } else {
      P = s.c;
      const int tt = (int)((unsigned)(i - big) / (unsigned)P);
      t = s.e + tt;
      j = i - big - tt * P;
    }
    *b0 = t * s.KB + even_lo(j, s.KB, P);
    *b1 = t * s.KB + even_lo(j + 1, s.KB, P);
  } else {
    *b0 = (i * s.a + (i < s.r ? i : s.r)) << s.qs;
    *b1 = *b0 + ((s.a + (i < s.r ? 1 : 0)) << s.qs);
  }
}

// The CTA whose run contains slab u (linear split).
__host__ __device__ __forceinline__ int gemm_split_owner_linear(const GemmSplit& s, int u) {
  u >>= s.qs;                         // its unit
  const int head = s.r * (s.a + 1);   // units of the longer runs
  return u < head ? (int)((unsigned)u / (unsigned)(s.a + 1)) : s.r + (int)((unsigned)(u - head) / (unsigned)s.a);
}

// Number of CTAs whose runs share tile t (the tile's combine waits for this many partials).
__host__ __device__ __forceinline__ int gemm_split_contributors(const GemmSplit& s, int t) {
  if (s.aligned) return t < s.e ? s.c + 1 : s.c;
  return gemm_split_owner_linear(s, t * s.KB + s.KB - 1) - gemm_split_owner_linear(s, t * s.KB) + 1;
}

}  // namespace w8a8

namespace w8a8 {

// ---------------------------------------------------------------- tensor-map TMA (2-D tile load)
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// L2 prefetches.  A prefetch is a hint: it changes no value that any later read returns (device
// memory is coherent in L2, and nothing lands in the SM), so it may be issued before a dependency
// wait on data that the previous kernel may still write.
// [src, src + bytes) into L2; src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// The L2 line holding addr.
__device__ __forceinline__ void prefetch_l2_line(const void* addr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(addr) : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
// Wait until the grids this one depends on have completed and their memory is visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid on the stream to begin launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace w8a8

namespace w8a8 {

// ---------------------------------------------------------------- global atomics with explicit ordering
// Fire-and-forget int32 add (no return value).
__device__ __forceinline__ void red_add_s32(int* addr, int v) {
  asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// Returning 64-bit add with no ordering beyond the word itself (no compiler memory barrier
// either: independent adds issue back to back).
__device__ __forceinline__ unsigned long long atom_add_relaxed_u64(unsigned long long* addr, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(addr), "l"(v));
  return old;
}

// Counter arrival: releases this thread's earlier writes (and, through a preceding warp barrier,
// its warp's) and acquires the writes released by earlier arrivals.
__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(uint32_t* addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

}  // namespace w8a8

namespace w8a8 {

// ---------------------------------------------------------------- fifth-generation tensor cores
// tcgen05 instructions (one CTA, cta_group::1).  Tensor memory addresses carry the lane in bits
// 31..16 and the 32-bit column in bits 15..0; a warp reaches lanes 32 * (warp % 4) ... + 31.

// Allocate `cols` tensor-memory columns (a power of two >= 32); the whole warp executes it and the
// base address lands in *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor: no swizzle, K-major.  Core matrix = 8 rows x 16 bytes; for a
// 16-bit operand, element (row r, k) sits at (r / 8) * sbo + (k / 8) * lbo + (r % 8) * 16 + (k % 8) * 2
// from the start address.  Bits 46..47 hold the descriptor version of this architecture (1).
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::f16: D f32 (bits 4..5 = 1), A and B f16 (0), both K-major,
// N / 8 in bits 17..22, M / 16 in bits 24..28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem_d] (+)= A[tmem_a] * B[desc_b]^T, A from tensor memory (lane = row, column c = the f16 pair
// k = 2c, 2c + 1), B from shared memory.  Issued by one thread.
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t desc_b, uint32_t idesc,
                                                bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          tmem_d),
      "r"(tmem_a), "l"(desc_b), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 16 consecutive columns of this thread's lane, written / read (warp-wide).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Four int8 values in offset binary, bytes in natural order (b0, b1, b2, b3) -> the fp16 pairs
// (b0, b1) and (b2, b3) (first element in the low half), exactly (see offset_bytes_to_half2).
__device__ __forceinline__ void offset_bytes_to_half2_pairs(uint32_t u, uint32_t& p01, uint32_t& p23) {
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  p01 = *reinterpret_cast<uint32_t*>(&ha);
  p23 = *reinterpret_cast<uint32_t*>(&hb);
}

}  // namespace w8a8
