// Internal host-side interfaces between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w8a8 {

// Every workspace starts with this header; its first 32-bit word is the device status.
constexpr size_t kWsHeaderBytes = 256;

// SMs of a GB300, the count assumed when no device can be queried (host-only plan queries).
constexpr int kDefaultSmCount = 152;

// Number of SMs of the current device, else kDefaultSmCount; clears any error the query raised.
int device_sm_count();

struct GemmPlan {
  int nt8, n_tiles, kb;
  long long slabs;
  int blocks, threads, stage_slabs, stages;
  int pack_f;   // split-tile combine: bits per element field of a two-element word (0: one per word)
  int split_unit;   // slabs per unit of a linear run split (1 or 4)
  size_t smem_bytes, workspace_bytes, partials_offset;
};

int gemm_plan(int M, int K, int N, int blocks, int sm_count, GemmPlan* plan);
// acc (optional): the exact int32 sums [M, N] are stored there as well.  stall: the test hook of
// W8A8_FLAG_TEST_STALL (one warp waits on a barrier that nothing completes, with a short bound).
cudaError_t gemm_launch(const GemmPlan& pl, const int8_t* x, const float* xs, const void* wp, const float* wsc,
                        void* out, int M, int K, int N, void* ws, bool pdl, cudaStream_t stream, int* acc = nullptr,
                        bool stall = false);

// M ranges of the two W8A8 arms: the register-fed decode kernel up to kDecodeMaxM rows, the
// tensor-memory (tcgen05) kernel above it up to kTcMaxM.
constexpr int kDecodeMaxM = 32;
constexpr int kTcMaxM = 128;

struct TcPlan {
  int mma_n;          // MMA N: activation rows covered (64 or 128)
  int tiles64;        // 64-row packed tiles of N
  int n_tiles;        // 128-row CTA tiles (pairs of packed tiles)
  int kb;             // K / 32
  long long units;    // n_tiles * kb: 32-k units of one CTA tile (the split's unit)
  int blocks, threads, stage_units, stages;
  size_t smem_bytes, workspace_bytes, counters_offset, partials_offset, x16_offset;
};

int tc_plan(int M, int K, int N, int blocks, int sm_count, TcPlan* plan);
cudaError_t tc_launch(const TcPlan& pl, const int8_t* x, const float* xs, const void* wp, const float* wsc, void* out,
                      int M, int K, int N, void* ws, bool pdl, cudaStream_t stream, int* acc = nullptr,
                      bool stall = false);

// Either arm.  M <= 32: the decode kernel.  M > 32: the tensor-memory kernel, or the decode kernel
// over consecutive row chunks of at most 32 (chunks > 1), whichever the measured cost model of
// any_plan predicts faster; an explicit CTA count (blocks > 0) or force_tc selects the
// tensor-memory kernel.
struct AnyPlan {
  bool tc;
  int chunks;      // decode launches: 1, or ceil(M / 32) row chunks for M > 32
  GemmPlan g;      // decode plan (of the 32-row chunks when chunks > 1)
  GemmPlan g_last; // chunks > 1: the plan of the last chunk's M - 32 (chunks - 1) rows
  TcPlan t;
  size_t workspace_bytes() const {
    if (tc) return t.workspace_bytes;
    return chunks > 1 && g_last.workspace_bytes > g.workspace_bytes ? g_last.workspace_bytes : g.workspace_bytes;
  }
};

int any_plan(int M, int K, int N, int blocks, int sm_count, AnyPlan* plan, bool force_tc = false);
cudaError_t any_launch(const AnyPlan& pl, const int8_t* x, const float* xs, const void* wp, const float* wsc, void* out,
                       int M, int K, int N, void* ws, bool pdl, cudaStream_t stream, int* acc = nullptr,
                       bool stall = false);
cudaError_t pack_launch(const int8_t* W, int K, int N, void* out, cudaStream_t stream);

struct Q8Plan {
  int n_tiles;       // 16-row tiles of N
  int kb;            // K / 32
  int warps;         // warps per CTA (each a contiguous run of k blocks)
  int splits;        // CTAs per tile along K (combined by the last arrival)
  int cluster;       // > 1: the tile's warps spread over a cluster of this many CTAs (splits == 1)
  int tile_warps;    // warps per tile (the k-block runs; equals warps unless cluster > 1)
  int blocks;        // n_tiles * splits * cluster
  size_t workspace_bytes, counters_offset, partials_offset;
};

int q8_plan(int T, int K, int N, Q8Plan* plan);
// gamma != NULL: the RMS-norm variant (norm weight gamma [K] bf16, epsilon eps).
cudaError_t q8_launch(const Q8Plan& pl, const void* x, const int8_t* q, const void* d, void* y, int T, int K, int N,
                      void* ws, bool pdl, cudaStream_t stream, const void* gamma = nullptr, float eps = 0.f);

// Encode a 2-D tiled tensor map through the driver entry point (no link-time libcuda dependency).
cudaError_t encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, void* base, const cuuint64_t* dims,
                                 const cuuint64_t* strides, const cuuint32_t* box, const cuuint32_t* estr,
                                 CUtensorMapSwizzle swizzle);

// Record a CUDA error (returns W8A8_ERR_CUDA) or a plain message as this thread's last error text.
int record_cuda_error(cudaError_t e, const char* where);
void record_error(const char* text);

// Raise a kernel's dynamic shared memory limit once per device.
cudaError_t ensure_smem_attribute(const void* kernel, int bytes);

}  // namespace w8a8
