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
