// w8a8_gemm_no_alloc: the W8A8 GEMM for callers that cannot allocate device memory.
//
// w8a8_gemm needs a caller-provided workspace (the split-tile accumulators).  Some callers have
// no way to provide one.  An inference plugin hosted inside another engine sees only the input and
// output pointers the host engine hands it, with no access to that engine's allocator.  A
// latency-critical request path may forbid cudaMalloc/cudaFree outright, because those calls can
// synchronise the device and stall every other stream.  For them this entry point runs the same
// kernel on a scratch area that lives in this library's own device memory: a file-scope __device__
// array reserved when the library's module is loaded on a device, and held there until the
// process exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/w8a8.h"
#include "internal.h"

namespace w8a8 {

// Largest workspace this entry point can serve: a plan needing more is rejected.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// The scratch area (zero when the module is loaded).  In host code this name is only a stand-in
// for the device symbol: its device address must be obtained with cudaGetSymbolAddress in each
// context that uses it (see scratch_in_current_context).
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

// Unique id of the current CUDA context (cuCtxGetId through the runtime's driver entry point, so
// the library needs no link-time libcuda).  Ids are never reused within a process, so a context
// created after cudaDeviceReset, or a context other than the device's primary one, gets its own
// cache entry.
static cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  static cudaError_t lookup = cudaSuccess;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    lookup = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q);
    if (lookup == cudaSuccess && q != cudaDriverEntryPointSuccess) lookup = cudaErrorSymbolNotFound;
    get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    if (lookup != cudaSuccess) return;
    fn = nullptr;
    lookup = cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q);
    if (lookup == cudaSuccess && q != cudaDriverEntryPointSuccess) lookup = cudaErrorSymbolNotFound;
    get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (lookup != cudaSuccess || !get_current || !get_id) return lookup != cudaSuccess ? lookup : cudaErrorSymbolNotFound;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!ctx) {
    *id = 0;   // no context current on this thread yet (the caller binds one, see below)
    return cudaSuccess;
  }
  if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// Device address of the scratch area in the current context: looked up once per context (the
// first call in a context, made before any stream capture) and cached.
static cudaError_t scratch_in_current_context(void** addr) {
  struct Entry {
    unsigned long long ctx;
    void* addr;
  };
  constexpr int kMaxContexts = 64;
  static Entry cache[kMaxContexts] = {};
  static int used = 0;
  static std::mutex mu;
  unsigned long long id = 0;
  cudaError_t e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (id != 0) {
    for (int i = 0; i < used; ++i)
      if (cache[i].ctx == id) {
        *addr = cache[i].addr;
        return cudaSuccess;
      }
  }
  // Set-up in this context: the runtime call below also binds the device's primary context to
  // this thread if none was current yet.
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
  if (e != cudaSuccess) return e;
  if (id == 0) {
    e = current_context_id(&id);
    if (e != cudaSuccess) return e;
  }
  if (id != 0 && used < kMaxContexts) cache[used++] = Entry{id, p};
  *addr = p;
  return cudaSuccess;
}

}  // namespace w8a8

using namespace w8a8;

extern "C" int w8a8_gemm_no_alloc(const int8_t* x_q, const float* x_scale, const void* W_packed,
                                  const float* w_scale, void* out, int M, int K, int N, int blocks,
                                  unsigned flags, void* stream) {
  if (!x_q || !x_scale || !W_packed || !w_scale || !out) return W8A8_ERR_INVALID_ARG;
  if (flags & ~(unsigned)(W8A8_FLAG_PDL | W8A8_FLAG_TENSOR_MEMORY_ARM | W8A8_FLAG_TEST_STALL))
    return W8A8_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  AnyPlan pl;
  const int rc = any_plan(M, K, N, blocks, sms, &pl, (flags & W8A8_FLAG_TENSOR_MEMORY_ARM) != 0);
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
  cudaError_t e = scratch_in_current_context(&ws);
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_gemm_no_alloc (scratch address)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The area keeps whatever the previous call left there.  Clear the regions this call relies on
  // being zero (the split-tile accumulators, counters and partial planes) before the kernel reads
  // them; the status word in the header is left alone (it collects device faults until
  // w8a8_gemm_no_alloc_status reads it), and the tensor-memory arm's fp16 activation copy, which
  // every such call rewrites, is not cleared.
  const size_t clear_end = pl.tc ? pl.t.x16_offset : pl.workspace_bytes();
  if (clear_end > kWsHeaderBytes) {
    e = cudaMemsetAsync(static_cast<uint8_t*>(ws) + kWsHeaderBytes, 0, clear_end - kWsHeaderBytes, s);
    if (e != cudaSuccess) return record_cuda_error(e, "w8a8_gemm_no_alloc (scratch clear)");
  }
  e = any_launch(pl, x_q, x_scale, W_packed, w_scale, out, M, K, N, ws, (flags & W8A8_FLAG_PDL) != 0, s, nullptr,
                 (flags & W8A8_FLAG_TEST_STALL) != 0);
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_gemm_no_alloc");
  return W8A8_OK;
}

extern "C" int w8a8_gemm_no_alloc_status(void* stream, uint32_t* status) {
  if (!status) return W8A8_ERR_INVALID_ARG;
  void* ws = nullptr;
  cudaError_t e = scratch_in_current_context(&ws);
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_gemm_no_alloc_status (scratch address)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(v), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_gemm_no_alloc_status");
  *status = v;
  return W8A8_OK;
}
