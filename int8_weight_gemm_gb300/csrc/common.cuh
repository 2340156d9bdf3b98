// Device building blocks shared by the kernels of this library (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/w8a8.h"

namespace w8a8 {

// A pipeline wait gives up after this many SM clock cycles (about one second at GB300 clocks) and
// reports W8A8_DEV_WAIT_TIMEOUT instead of spinning forever.  The cycle counter is cheap to read;
// it is consulted only every 64 unsuccessful polls.
constexpr long long kWaitTimeoutCycles = 2000000000ll;

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

// Wait for the phase of `parity` to complete.  Bounded: gives up when another thread of the CTA
// has raised *abort, or after kWaitTimeoutCycles (then records the timeout in *status and raises
// *abort).  Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > kWaitTimeoutCycles) {
        atomicOr(status, W8A8_DEV_WAIT_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// Wait for a phase that is sure to complete (copies already issued): bounded by the cycle limit
// only.  Returns false on timeout (recorded in *status).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint32_t* status) {
  const long long t0 = clock64();
  for (unsigned it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && clock64() - t0 > kWaitTimeoutCycles) {
      atomicOr(status, W8A8_DEV_WAIT_TIMEOUT);
      return false;
    }
  }
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

// ---------------------------------------------------------------- split plan (host and device)
// CTA i of G owns slabs [split_lo(i), split_lo(i+1)) of U: equal runs within one slab.
__host__ __device__ __forceinline__ long long split_lo(long long i, long long U, long long G) {
  return i * U / G;
}

// The CTA whose run contains slab u (requires G <= U, so that no run is empty).
__host__ __device__ __forceinline__ long long split_owner(long long u, long long U, long long G) {
  return ((u + 1) * G + U - 1) / U - 1;
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
