// C ABI of the library: argument checks, launch plans and error reporting.  Every check runs
// before any launch; each compute entry point issues one kernel launch (two for w8a8_gemm with
// M > 32: the fp16 activation copy, then the GEMM as its programmatic dependent) and nothing else.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/w8a8.h"
#include "common.cuh"
#include "internal.h"

namespace w8a8 {

static thread_local char g_last_error[256] = "";

static int cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
  return W8A8_ERR_CUDA;
}

int record_cuda_error(cudaError_t e, const char* where) { return cuda_fail(e, where); }

void record_error(const char* text) { std::snprintf(g_last_error, sizeof(g_last_error), "%s", text); }

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The GB300 count when no device can be queried, so that the host-only plan queries answer the
// same way on a machine without a GPU.
int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return kDefaultSmCount;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return kDefaultSmCount;
  }
  return sms;
}

cudaError_t ensure_smem_attribute(const void* kernel, int bytes) {
  // One record per (kernel, device); a small fixed table is plenty for this library's kernels.
  struct Entry {
    const void* k;
    int dev;
    int bytes;
  };
  static Entry table[64];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].k == kernel && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (used < 64) table[used++] = Entry{kernel, dev, bytes};
  return cudaSuccess;
}

cudaError_t encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, void* base, const cuuint64_t* dims,
                                 const cuuint64_t* strides, const cuuint32_t* box, const cuuint32_t* estr,
                                 CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  static cudaError_t lookup = cudaSuccess;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    void* fn = nullptr;
    lookup = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (lookup == cudaSuccess && q != cudaDriverEntryPointSuccess) lookup = cudaErrorSymbolNotFound;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (lookup != cudaSuccess || !encode) return lookup != cudaSuccess ? lookup : cudaErrorSymbolNotFound;
  CUresult r = encode(map, type, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Cost model of the two ways to run 32 < M <= 128: least-squares lines through graph-replay
// timings on GB300 (cold weights, 152 SMs) of both kernels over six weight shapes from 6 to 96 MiB
// (K x N = 4096 x 1536, 4096 x 2560, 2048 x 4096, 4096 x 8192, 12288 x 4096, 4096 x 24576), the
// decode kernel at M = 8, 16, 24, 32 and the tensor-memory kernel at M = 48 ... 128: each call
// costs a fixed part plus a part proportional to the packed weight's size, by decode n8-tile count
// and by the tensor-memory kernel's MMA width.  The decode kernel's per-byte cost grows with M (its
// MMA and activation-conversion work per weight byte do), the tensor-memory kernel's much less, so
// row chunks win on small weights and the tensor-memory kernel on large ones.  The decode lines fit
// within 8 %; the tensor-memory kernel's times depend on how its tiles fall over the SMs and fit
// only within 22 %, yet on the 24 measured (shape, M) points the lines pick the faster arm every
// time (fitted again after the decode launches became programmatic dependents and the
// tensor-memory converters moved to stage groups).
static double decode_cost_us(int nt8, double w_mib) {
  static const double fixed[5] = {0.0, 3.18, 3.97, 3.87, 4.19}, per_mib[5] = {0.0, 0.150, 0.164, 0.267, 0.306};
  return fixed[nt8] + per_mib[nt8] * w_mib;
}
static double tc_cost_us(int M, double w_mib) { return M <= 64 ? 17.28 + 0.422 * w_mib : 27.75 + 0.463 * w_mib; }

int any_plan(int M, int K, int N, int blocks, int sm_count, AnyPlan* plan, bool force_tc) {
  plan->tc = false;
  plan->chunks = 1;
  if (M <= kDecodeMaxM) return gemm_plan(M, K, N, blocks, sm_count, &plan->g);
  int rc = tc_plan(M, K, N, blocks, sm_count, &plan->t);
  if (rc != W8A8_OK) return rc;
  plan->tc = true;
  if (force_tc || blocks > 0) return W8A8_OK;
  const int chunks = (M + kDecodeMaxM - 1) / kDecodeMaxM;
  const int last = M - kDecodeMaxM * (chunks - 1);
  const double w_mib = (double)((N + 63) / 64) * 64.0 * (double)K / 1048576.0;
  const double t_chunks = (chunks - 1) * decode_cost_us(4, w_mib) + decode_cost_us((last + 7) / 8, w_mib);
  if (t_chunks >= tc_cost_us(M, w_mib)) return W8A8_OK;
  if ((rc = gemm_plan(kDecodeMaxM, K, N, 0, sm_count, &plan->g)) != W8A8_OK) return rc;
  if ((rc = gemm_plan(last, K, N, 0, sm_count, &plan->g_last)) != W8A8_OK) return rc;
  plan->tc = false;
  plan->chunks = chunks;
  return W8A8_OK;
}

cudaError_t any_launch(const AnyPlan& pl, const int8_t* x, const float* xs, const void* wp, const float* wsc, void* out,
                       int M, int K, int N, void* ws, bool pdl, cudaStream_t stream, int* acc, bool stall) {
  if (pl.tc) return tc_launch(pl.t, x, xs, wp, wsc, out, M, K, N, ws, pdl, stream, acc, stall);
  if (pl.chunks == 1) return gemm_launch(pl.g, x, xs, wp, wsc, out, M, K, N, ws, pdl, stream, acc, stall);
  // Row chunks, one decode launch each, in stream order on the one workspace (each call leaves it
  // zeroed for the next).  With PDL each chunk's weight prefetch overlaps the previous chunk's tail.
  for (int c = 0; c < pl.chunks; ++c) {
    const int m0 = kDecodeMaxM * c;
    const int rows = c + 1 < pl.chunks ? kDecodeMaxM : M - m0;
    const GemmPlan& g = c + 1 < pl.chunks ? pl.g : pl.g_last;
    cudaError_t e = gemm_launch(g, x + (size_t)m0 * K, xs + m0, wp, wsc, static_cast<uint16_t*>(out) + (size_t)m0 * N,
                                rows, K, N, ws, pdl, stream, acc ? acc + (size_t)m0 * N : nullptr, stall && c == 0);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace w8a8

using namespace w8a8;

extern "C" {

int w8a8_version(void) { return 100; }

const char* w8a8_status_string(int status) {
  switch (status) {
    case W8A8_OK: return "ok";
    case W8A8_ERR_INVALID_ARG: return "invalid argument";
    case W8A8_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case W8A8_ERR_MISALIGNED: return "misaligned pointer";
    case W8A8_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case W8A8_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* w8a8_last_error(void) { return g_last_error; }

int w8a8_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes == 0) return W8A8_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return W8A8_ERR_MISALIGNED;
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "w8a8_workspace_init");
  return W8A8_OK;
}

int w8a8_workspace_status(void* ws, size_t ws_bytes, void* stream, uint32_t* status) {
  if (!ws || !status || ws_bytes < kWsHeaderBytes) return W8A8_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return W8A8_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(v), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "w8a8_workspace_status");
  *status = v;
  return W8A8_OK;
}

size_t w8a8_packed_weight_bytes(int K, int N) {
  if (K < 1 || N < 1) return 0;
  return (size_t)((N + 63) / 64) * 64 * (size_t)K;
}

size_t w8a8_workspace_bytes(int M_max, int K, int N, int blocks) {
  if (M_max < 1 || M_max > kTcMaxM) return 0;
  const int sms = device_sm_count();
  size_t best = 0;
  // One plan per kernel variant that some M in [1, M_max] runs: the decode arm's n8-tile counts,
  // then the tensor-memory arm's two MMA widths.
  // For M > 32 the tensor-memory arm's plan is taken whether or not the automatic plan picks it
  // (the decode arm's row chunks need no more than its M = 32 plan, probed here as well).
  const int probes[] = {1, 9, 17, 25, 32, 33, 64, 65, 128};
  for (int m : probes) {
    if (m > M_max) break;
    AnyPlan pl;
    if (any_plan(m, K, N, blocks, sms, &pl, true) != W8A8_OK) return 0;
    if (pl.workspace_bytes() > best) best = pl.workspace_bytes();
  }
  AnyPlan pl;
  if (any_plan(M_max, K, N, blocks, sms, &pl, true) != W8A8_OK) return 0;
  return pl.workspace_bytes() > best ? pl.workspace_bytes() : best;
}

int w8a8_plan(int M, int K, int N, int blocks, w8a8_plan_t* plan) { return w8a8_plan_flags(M, K, N, blocks, 0u, plan); }

int w8a8_plan_flags(int M, int K, int N, int blocks, unsigned flags, w8a8_plan_t* plan) {
  if (!plan) return W8A8_ERR_INVALID_ARG;
  if (flags & ~(unsigned)(W8A8_FLAG_PDL | W8A8_FLAG_TENSOR_MEMORY_ARM | W8A8_FLAG_TEST_STALL))
    return W8A8_ERR_INVALID_ARG;
  AnyPlan ap;
  int rc = any_plan(M, K, N, blocks, device_sm_count(), &ap, (flags & W8A8_FLAG_TENSOR_MEMORY_ARM) != 0);
  if (rc != W8A8_OK) return rc;
  if (ap.tc) {
    const TcPlan& pl = ap.t;
    plan->n8_tiles = pl.mma_n / 8;
    plan->n_tiles = pl.n_tiles;
    plan->k_blocks = pl.kb;
    plan->slabs = pl.units;
    plan->blocks = pl.blocks;
    plan->threads = pl.threads;
    plan->stage_slabs = pl.stage_units;
    plan->stages = pl.stages;
    plan->smem_bytes = pl.smem_bytes;
    plan->workspace_bytes = pl.workspace_bytes;
    plan->combine_pack_bits = 0;
    plan->tile_rows = 128;
    plan->tensor_memory = 1;
    plan->row_chunks = 1;
    plan->split_unit = 1;
    return W8A8_OK;
  }
  const GemmPlan& pl = ap.g;
  plan->n8_tiles = pl.nt8;
  plan->n_tiles = pl.n_tiles;
  plan->k_blocks = pl.kb;
  plan->slabs = pl.slabs;
  plan->blocks = pl.blocks;
  plan->threads = pl.threads;
  plan->stage_slabs = pl.stage_slabs;
  plan->stages = pl.stages;
  plan->smem_bytes = pl.smem_bytes;
  plan->workspace_bytes = pl.workspace_bytes;
  plan->combine_pack_bits = pl.pack_f;
  plan->tile_rows = 64;
  plan->tensor_memory = 0;
  plan->row_chunks = ap.chunks;
  plan->split_unit = pl.split_unit;
  return W8A8_OK;
}

int w8a8_split_bounds_m(int M, int K, int N, int blocks, long long* bounds, int n_bounds) {
  if (!bounds) return W8A8_ERR_INVALID_ARG;
  AnyPlan ap;
  int rc = any_plan(M, K, N, blocks, device_sm_count(), &ap);
  if (rc != W8A8_OK) return rc;
  const int n_tiles = ap.tc ? ap.t.n_tiles : ap.g.n_tiles;
  const int kb = ap.tc ? ap.t.kb : ap.g.kb;
  const int g = ap.tc ? ap.t.blocks : ap.g.blocks;
  if (n_bounds != g + 1) return W8A8_ERR_INVALID_ARG;
  const GemmSplit sp = make_gemm_split(n_tiles, kb, g, !ap.tc);
  for (int i = 0; i < g; ++i) {
    int b0, b1;
    gemm_split_run(sp, i, &b0, &b1);
    bounds[i] = b0;
  }
  bounds[g] = (long long)n_tiles * kb;
  return W8A8_OK;
}

int w8a8_split_bounds(int K, int N, int blocks, long long* bounds, int n_bounds) {
  return w8a8_split_bounds_m(1, K, N, blocks, bounds, n_bounds);
}

int w8a8_pack_weights(const int8_t* W, int K, int N, void* W_packed, void* ws, size_t ws_bytes, void* stream) {
  if (!W || !W_packed) return W8A8_ERR_INVALID_ARG;
  if (K < 1 || K > 65536 || N < 1 || N > 1048576) return W8A8_ERR_INVALID_ARG;
  if (K % 32 != 0 || N % 8 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_packed, 16)) return W8A8_ERR_MISALIGNED;
  if (ws) {
    int rc = w8a8_workspace_init(ws, ws_bytes, stream);
    if (rc != W8A8_OK) return rc;
  }
  cudaError_t e = pack_launch(W, K, N, W_packed, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "w8a8_pack_weights");
  return W8A8_OK;
}

// w8a8_gemm and w8a8_gemm_acc: every check, then the launch (acc may be NULL).
static int gemm_call(const char* name, const int8_t* x_q, const float* x_scale, const void* W_packed,
                     const float* w_scale, void* out, int32_t* acc, int M, int K, int N, int blocks, unsigned flags,
                     void* ws, size_t ws_bytes, void* stream) {
  if (!x_q || !x_scale || !W_packed || !w_scale || !out || !ws) return W8A8_ERR_INVALID_ARG;
  if (flags & ~(unsigned)(W8A8_FLAG_PDL | W8A8_FLAG_TENSOR_MEMORY_ARM | W8A8_FLAG_TEST_STALL))
    return W8A8_ERR_INVALID_ARG;
  AnyPlan pl;
  int rc = any_plan(M, K, N, blocks, device_sm_count(), &pl, (flags & W8A8_FLAG_TENSOR_MEMORY_ARM) != 0);
  if (rc != W8A8_OK) return rc;
  if (!aligned(x_q, 16) || !aligned(W_packed, 16) || !aligned(out, 16) || !aligned(x_scale, 4) ||
      !aligned(w_scale, 4) || !aligned(ws, 256) || !aligned(acc, 4))
    return W8A8_ERR_MISALIGNED;
  if (ws_bytes < pl.workspace_bytes()) return W8A8_ERR_WORKSPACE_TOO_SMALL;
  cudaError_t e = any_launch(pl, x_q, x_scale, W_packed, w_scale, out, M, K, N, ws, (flags & W8A8_FLAG_PDL) != 0,
                             static_cast<cudaStream_t>(stream), acc, (flags & W8A8_FLAG_TEST_STALL) != 0);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return W8A8_OK;
}

int w8a8_gemm(const int8_t* x_q, const float* x_scale, const void* W_packed, const float* w_scale, void* out,
              int M, int K, int N, int blocks, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  return gemm_call("w8a8_gemm", x_q, x_scale, W_packed, w_scale, out, nullptr, M, K, N, blocks, flags, ws, ws_bytes,
                   stream);
}

int w8a8_gemm_acc(const int8_t* x_q, const float* x_scale, const void* W_packed, const float* w_scale, void* out,
                  int32_t* acc, int M, int K, int N, int blocks, unsigned flags, void* ws, size_t ws_bytes,
                  void* stream) {
  if (!acc) return W8A8_ERR_INVALID_ARG;
  return gemm_call("w8a8_gemm_acc", x_q, x_scale, W_packed, w_scale, out, acc, M, K, N, blocks, flags, ws, ws_bytes,
                   stream);
}

size_t q8_0_workspace_bytes(int T_max, int K, int N) {
  Q8Plan pl;
  if (q8_plan(T_max, K, N, &pl) != W8A8_OK) return 0;
  return pl.workspace_bytes;
}

int q8_0_gemv(const void* x, const int8_t* q, const void* d, void* y, int T, int K, int N, unsigned flags, void* ws,
              size_t ws_bytes, void* stream) {
  if (!x || !q || !d || !y || !ws) return W8A8_ERR_INVALID_ARG;
  if (flags & ~(unsigned)W8A8_FLAG_PDL) return W8A8_ERR_INVALID_ARG;
  Q8Plan pl;
  int rc = q8_plan(T, K, N, &pl);
  if (rc != W8A8_OK) return rc;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(d, 2) || !aligned(y, 2) || !aligned(ws, 256))
    return W8A8_ERR_MISALIGNED;
  if (ws_bytes < pl.workspace_bytes) return W8A8_ERR_WORKSPACE_TOO_SMALL;
  cudaError_t e = q8_launch(pl, x, q, d, y, T, K, N, ws, (flags & W8A8_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "q8_0_gemv");
  return W8A8_OK;
}

int q8_0_gemv_rms(const void* x, const void* gamma, float eps, const int8_t* q, const void* d, void* y, int T, int K,
                  int N, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
  if (!x || !gamma || !q || !d || !y || !ws) return W8A8_ERR_INVALID_ARG;
  if (flags & ~(unsigned)W8A8_FLAG_PDL) return W8A8_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !(eps <= 3.0e38f)) return W8A8_ERR_INVALID_ARG;   // finite, not negative (NaN fails too)
  Q8Plan pl;
  int rc = q8_plan(T, K, N, &pl);
  if (rc != W8A8_OK) return rc;
  if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(q, 16) || !aligned(d, 2) || !aligned(y, 2) ||
      !aligned(ws, 256))
    return W8A8_ERR_MISALIGNED;
  if (ws_bytes < pl.workspace_bytes) return W8A8_ERR_WORKSPACE_TOO_SMALL;
  cudaError_t e = q8_launch(pl, x, q, d, y, T, K, N, ws, (flags & W8A8_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream),
                            gamma, eps);
  if (e != cudaSuccess) return cuda_fail(e, "q8_0_gemv_rms");
  return W8A8_OK;
}

}  // extern "C"
