// Read-only bandwidth probe: the achievable HBM read rate that the weight stream is measured
// against.  A plain grid-stride read of 16-byte vectors through the non-coherent path, four loads
// in flight per thread per iteration, XOR-reduced so that no load can be dropped; the reduction is
// written only if it equals a value no real buffer produces in practice.  Nothing of the GEMM or
// the Q8_0 read runs here.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/w8a8.h"
#include "internal.h"

namespace w8a8 {

__global__ void __launch_bounds__(512) read_probe_kernel(const uint4* __restrict__ p, size_t n16,
                                                         unsigned long long* sink) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldg(p + i), b = __ldg(p + i + stride), c = __ldg(p + i + 2 * stride),
                d = __ldg(p + i + 3 * stride);
    acc ^= (a.x ^ a.y ^ a.z ^ a.w) ^ (b.x ^ b.y ^ b.z ^ b.w) ^ (c.x ^ c.y ^ c.z ^ c.w) ^ (d.x ^ d.y ^ d.z ^ d.w);
  }
  for (; i < n16; i += stride) {
    const uint4 a = __ldg(p + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  if (acc == 0x9E3779B9u) atomicAdd(sink, 1ull);
}

}  // namespace w8a8

using namespace w8a8;

extern "C" int w8a8_read_probe(const void* buf, size_t bytes, void* sink, void* stream) {
  if (!buf || !sink || bytes < 16) return W8A8_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(buf) & 15u) || (reinterpret_cast<uintptr_t>(sink) & 7u)) return W8A8_ERR_MISALIGNED;
  const int sms = device_sm_count();
  // Two 512-thread CTAs per SM: 32 warps per SM, each with four 16-byte loads per lane in flight.
  read_probe_kernel<<<2 * sms, 512, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(buf), bytes / 16, static_cast<unsigned long long*>(sink));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_read_probe");
  return W8A8_OK;
}

// ---------------------------------------------------------------------------------------------
// Tensor-pipe rate probe: the two register-fed MMA forms the decode kernel could use for its int8
// products, timed by the caller.  Each warp runs `iters` rounds of eight independent MMAs (eight
// accumulator sets, so the pipe never waits on a result) on operands that change every round; the
// accumulators are folded into a value written only in a case real runs never produce.
//  kind 0: mma.sync m16n8k16 f16 x f16 -> f32 (the form the decode kernel uses, after converting
//          int8 to fp16 exactly): 2 * 16 * 8 * 16 = 4096 flops per MMA.
//  kind 1: mma.sync m16n8k32 s8 x s8 -> s32: 2 * 16 * 8 * 32 = 8192 int ops per MMA.
// ---------------------------------------------------------------------------------------------
namespace w8a8 {

template <int KIND>
__global__ void __launch_bounds__(256) mma_rate_kernel(int iters, unsigned long long* sink) {
  const uint32_t lane = threadIdx.x & 31;
  uint32_t a0 = 0x3C003C00u ^ lane, a1 = 0x3C013C01u ^ lane, a2 = 0x3C023C02u, a3 = 0x3C033C03u;
  uint32_t b0 = 0x3C003C00u ^ (lane << 1), b1 = 0x3C043C04u;
  float f[8][4] = {};
  int s[8][4] = {};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (KIND == 0) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(f[r][0]), "+f"(f[r][1]), "+f"(f[r][2]), "+f"(f[r][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      } else {
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+r"(s[r][0]), "+r"(s[r][1]), "+r"(s[r][2]), "+r"(s[r][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      }
    }
    a0 += 0x00010001u;
    b1 ^= (uint32_t)it;
  }
  uint32_t acc = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc ^= __float_as_uint(f[r][c]) ^ (uint32_t)s[r][c];
  if (acc == 0x9E3779B9u) atomicAdd(sink, 1ull);
}

}  // namespace w8a8

extern "C" int w8a8_mma_rate_probe(int kind, int iters, void* sink, void* stream) {
  if ((kind != 0 && kind != 1) || iters < 1 || iters > (1 << 24) || !sink) return W8A8_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(sink) & 7u) return W8A8_ERR_MISALIGNED;
  const int sms = device_sm_count();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long* k = static_cast<unsigned long long*>(sink);
  // Two CTAs of eight warps per SM: four warps per sub-partition, as many as the decode kernel runs.
  if (kind == 0) mma_rate_kernel<0><<<2 * sms, 256, 0, s>>>(iters, k);
  else mma_rate_kernel<1><<<2 * sms, 256, 0, s>>>(iters, k);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_mma_rate_probe");
  return W8A8_OK;
}
