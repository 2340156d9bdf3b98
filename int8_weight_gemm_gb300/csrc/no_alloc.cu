// w8a8_gemm_no_alloc: the W8A8 GEMM for callers that cannot allocate device memory.
//
// w8a8_gemm needs a caller-provided workspace (the split-tile accumulators).  Some callers have
// no way to provide one.  An inference plugin hosted inside another engine sees only the input and
// output pointers the host engine hands it, with no access to that engine's allocator.  A latency-critical request path may forbid cudaMalloc/cudaFree
// outright, because those calls can synchronise the device and stall every other stream.  For
// them this entry point runs the same kernel on a scratch area that lives in this library's own
// device memory: a file-scope __device__ array reserved when the library's module is loaded on a
// device, and held there until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/w8a8.h"
#include "internal.h"

namespace w8a8 {

// Largest workspace this entry point can serve: a plan needing more is rejected.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// The scratch area.  In host code this name is only a stand-in for the device symbol: its device
// address must be obtained with cudaGetSymbolAddress on each device (see scratch_on_current_device).
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch area on the current device, looked up once per device and cached.
static cudaError_t scratch_on_current_device(void** addr) {
  constexpr int kMaxDevices = 64;
  static void* cache[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess) return e;
    cache[dev] = p;
  }
  *addr = cache[dev];
  return cudaSuccess;
}

}  // namespace w8a8

using namespace w8a8;

extern "C" int w8a8_gemm_no_alloc(const int8_t* x_q, const float* x_scale, const void* W_packed,
                                  const float* w_scale, void* out, int M, int K, int N, int blocks,
                                  unsigned flags, void* stream) {
  if (!x_q || !x_scale || !W_packed || !w_scale || !out) return W8A8_ERR_INVALID_ARG;
  if (flags & ~(unsigned)W8A8_FLAG_PDL) return W8A8_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  AnyPlan pl;
  const int rc = any_plan(M, K, N, blocks, sms, &pl);
  if (rc != W8A8_OK) return rc;
  auto misaligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (misaligned(x_q, 16) || misaligned(W_packed, 16) || misaligned(out, 16) || misaligned(x_scale, 4) ||
      misaligned(w_scale, 4))
    return W8A8_ERR_MISALIGNED;
  if (pl.workspace_bytes() > kNoAllocScratchBytes) {
    record_error("w8a8_gemm_no_alloc: this shape needs more scratch than the built-in 16 MiB area");
    return W8A8_ERR_WORKSPACE_TOO_SMALL;
  }
  void* ws = nullptr;
  cudaError_t e = scratch_on_current_device(&ws);
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_gemm_no_alloc (scratch address)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The area keeps whatever the previous call left there: clear the part this call relies on
  // (status word and split-tile accumulators) before the kernel reads it.
  e = cudaMemsetAsync(ws, 0, pl.workspace_bytes(), s);
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_gemm_no_alloc (scratch clear)");
  e = any_launch(pl, x_q, x_scale, W_packed, w_scale, out, M, K, N, ws, (flags & W8A8_FLAG_PDL) != 0, s);
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_gemm_no_alloc");
  return W8A8_OK;
}
