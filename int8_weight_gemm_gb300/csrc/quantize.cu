// Quantisation around the two operators: the W8A8 GEMM's int8 activations and per-row scales,
// Q8_0 weights from BF16 at load, and the re-layout between ggml's 34-byte Q8_0 blocks and the
// split layout the Q8_0 read takes.
//
// Sources:
//  * "sycl: STRATA_HC_Q8=1 reads the Q8_0 hyper-connection projections", section "What changed",
//    the loader bullet: BF16 tensors are quantised with ggml's rounding, d = amax / 127 stored as
//    fp16 and q = round(x / d), and uploaded in the split layout ("the same bytes as ggml's 34-byte
//    blocks, reordered").
//  * "INT8 W8A8 GEMM - Decode (M <= 32) - gfx928 / SGLang TP4", operator line: x_q[M,K] int8 with
//    x_scale[M,1]; the timed GEMM excludes the quantisation.
// Readings where the pages are silent: amax over a 32-value block (Q8_0) or over a row (the
// activations); x divided by the float32 scale (before any fp16 storage); C's roundf (halves away
// from zero); a zero block or row gets scale 0 and quants 0.  Every step is a single IEEE
// operation (division and fp16 conversion round to nearest even, roundf is exact), so the results
// are bit-identical to a scalar CPU evaluation.
//
// All three kernels move a few MB at most and are bound by HBM (or by launch latency at decode
// sizes): 16-byte loads, 8- or 16-byte stores, no shared-memory staging beyond one reduction.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/w8a8.h"
#include "internal.h"

namespace w8a8 {

constexpr int kRowThreads = 256;

// The eight bf16 values of a 16-byte vector as floats (exact).
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// q = roundf(x / s) for eight values, packed little-endian into two words (s != 0).
__device__ __forceinline__ uint2 quantize8(const float (&f)[8], float s) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int qi = s == 0.0f ? 0 : (int)roundf(__fdiv_rn(f[i], s));
    w[i >> 2] |= ((uint32_t)qi & 0xFFu) << (8 * (i & 3));
  }
  return make_uint2(w[0], w[1]);
}

// One CTA per activation row: the row's amax (first pass), then its quants (second pass, the row
// is L2-resident by then).
__global__ void __launch_bounds__(kRowThreads) quantize_rows_kernel(const uint4* __restrict__ x, uint2* __restrict__ xq,
                                                                    float* __restrict__ xs, int K) {
  __shared__ float red[kRowThreads / 32];
  // A programmatic dependent launched after this grid (every decode GEMM launch is one) may start
  // now: it prefetches its weights into L2 meanwhile, and waits for this grid to complete before
  // it reads x_q or x_scale.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int row = blockIdx.x;
  const int nv = K / 8;
  const uint4* src = x + (size_t)row * nv;
  float amax = 0.0f;
  for (int i = threadIdx.x; i < nv; i += kRowThreads) {
    float f[8];
    bf16x8_to_f32(__ldg(src + i), f);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kRowThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float s = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) xs[row] = s;
  uint2* dst = xq + (size_t)row * nv;
  for (int i = threadIdx.x; i < nv; i += kRowThreads) {
    float f[8];
    bf16x8_to_f32(__ldg(src + i), f);
    dst[i] = quantize8(f, s);
  }
}

// Q8_0 from BF16: four consecutive threads hold the 32 values of one block (8 each), so a
// block's amax is two lane exchanges away; the first of the four stores the fp16 scale.
__global__ void __launch_bounds__(256) q8_0_quantize_kernel(const uint4* __restrict__ w, uint2* __restrict__ q,
                                                            uint16_t* __restrict__ d, long long chunks) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  // Every thread of a warp runs the same number of iterations (chunks is a multiple of 4 and the
  // stride a multiple of 32), so the shuffles below always see the whole warp's lanes of a block.
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c - (threadIdx.x & 31) < chunks; c += stride) {
    const bool live = c < chunks;
    float f[8];
    bf16x8_to_f32(live ? __ldg(w + c) : make_uint4(0u, 0u, 0u, 0u), f);
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float s = __fdiv_rn(amax, 127.0f);
    if (live) {
      q[c] = quantize8(f, s);
      if ((c & 3) == 0) d[c >> 2] = __half_as_ushort(__float2half_rn(s));
    }
  }
}

// ggml blocks (per block: fp16 scale, then 32 quants; 34 bytes, 2-byte aligned) -> split layout.
__global__ void __launch_bounds__(256) q8_0_split_from_blocks_kernel(const uint16_t* __restrict__ blocks,
                                                                     uint4* __restrict__ q, uint16_t* __restrict__ d,
                                                                     long long nblocks) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    const uint16_t* src = blocks + b * 17;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (uint32_t)__ldg(src + 1 + 2 * i) | ((uint32_t)__ldg(src + 2 + 2 * i) << 16);
    d[b] = __ldg(src);
    q[2 * b] = make_uint4(w[0], w[1], w[2], w[3]);
    q[2 * b + 1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// Split layout -> ggml blocks.
__global__ void __launch_bounds__(256) q8_0_blocks_from_split_kernel(const uint4* __restrict__ q,
                                                                     const uint16_t* __restrict__ d,
                                                                     uint16_t* __restrict__ blocks, long long nblocks) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    const uint4 a = __ldg(q + 2 * b), c = __ldg(q + 2 * b + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
    uint16_t* dst = blocks + b * 17;
    dst[0] = __ldg(d + b);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      dst[1 + 2 * i] = (uint16_t)(w[i] & 0xFFFFu);
      dst[2 + 2 * i] = (uint16_t)(w[i] >> 16);
    }
  }
}

static unsigned grid_for(long long items, int threads) {
  long long g = (items + threads - 1) / threads;
  const long long cap = 64LL * kDefaultSmCount;   // grid-stride beyond a few waves
  if (g > cap) g = cap;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace w8a8

using namespace w8a8;

static bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

extern "C" int w8a8_quantize_activations(const void* x, int8_t* x_q, float* x_scale, int M, int K, void* stream) {
  if (!x || !x_q || !x_scale || M < 1 || M > (1 << 20) || K < 8 || K > 65536) return W8A8_ERR_INVALID_ARG;
  if (K % 8 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
  if (misaligned(x, 16) || misaligned(x_q, 8) || misaligned(x_scale, 4)) return W8A8_ERR_MISALIGNED;
  quantize_rows_kernel<<<(unsigned)M, kRowThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(x), reinterpret_cast<uint2*>(x_q), x_scale, K);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "w8a8_quantize_activations");
  return W8A8_OK;
}

extern "C" int q8_0_quantize(const void* w, int8_t* q, void* d, int K, int N, void* stream) {
  if (!w || !q || !d || K < 32 || K > 65536 || N < 1 || N > 1048576) return W8A8_ERR_INVALID_ARG;
  if (K % 32 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
  if (misaligned(w, 16) || misaligned(q, 8) || misaligned(d, 2)) return W8A8_ERR_MISALIGNED;
  const long long chunks = (long long)N * K / 8;
  q8_0_quantize_kernel<<<grid_for(chunks, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(w), reinterpret_cast<uint2*>(q), static_cast<uint16_t*>(d), chunks);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "q8_0_quantize");
  return W8A8_OK;
}

extern "C" int q8_0_split_from_blocks(const void* blocks, int8_t* q, void* d, int K, int N, void* stream) {
  if (!blocks || !q || !d || K < 32 || K > 65536 || N < 1 || N > 1048576) return W8A8_ERR_INVALID_ARG;
  if (K % 32 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
  if (misaligned(blocks, 2) || misaligned(q, 16) || misaligned(d, 2)) return W8A8_ERR_MISALIGNED;
  const long long nblocks = (long long)N * (K / 32);
  q8_0_split_from_blocks_kernel<<<grid_for(nblocks, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(blocks), reinterpret_cast<uint4*>(q), static_cast<uint16_t*>(d), nblocks);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "q8_0_split_from_blocks");
  return W8A8_OK;
}

extern "C" int q8_0_blocks_from_split(const int8_t* q, const void* d, void* blocks, int K, int N, void* stream) {
  if (!blocks || !q || !d || K < 32 || K > 65536 || N < 1 || N > 1048576) return W8A8_ERR_INVALID_ARG;
  if (K % 32 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
  if (misaligned(blocks, 2) || misaligned(q, 16) || misaligned(d, 2)) return W8A8_ERR_MISALIGNED;
  const long long nblocks = (long long)N * (K / 32);
  q8_0_blocks_from_split_kernel<<<grid_for(nblocks, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(q), static_cast<const uint16_t*>(d), static_cast<uint16_t*>(blocks), nblocks);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e, "q8_0_blocks_from_split");
  return W8A8_OK;
}
