// Q8_0 weight GEMV for sm_103a: y[T,N] = x[T,K] (bf16) times Q8_0 weights, T <= 8, bf16 out.
//
// Operator: "sycl: STRATA_HC_Q8=1 reads the Q8_0 hyper-connection projections", section "What
// changed": Q8_0 blocks of 32 int8 quants along K with one fp16 scale, the split layout (all
// quants row-major, then all scales), fixed-order partial sums, and for the long-K shape a last
// work-group combine through an atomic counter that never waits and is reset by the last arrival.
//
// GB300 mapping: one warp owns a 16-row tile of N over a contiguous run of 32-k blocks and
// multiplies it on the bf16 tensor path (mma.sync m16n8k16): the quants convert exactly to bf16,
// the activations are bf16 already, and the T <= 8 activation rows are the MMA's n8 columns.
// Each block's 16x8 product is scaled by its fp16 scale d and added in fp32, block by block in
// ascending k.  Warps of a CTA split the CTA's k range into contiguous runs and are summed in warp
// order through shared memory; when K is long the CTAs of one tile are combined by the last to
// arrive, in ascending split order.  Every order is fixed, so replays are bit-identical.
//
// RMS-norm variant (q8_0_gemv_rms): the same page's down kernel stages R' * w_norm unscaled with
// the rows' sums of squares, and the last work-group to arrive applies rs per stream.  Here each
// lane multiplies its activations by the norm weight g as it loads them (bf16 x bf16 is exact in
// fp32, rounded once to bf16 for the MMA) and sums their squares in fp32; the squares travel with
// the dot products through every combine (warp order, the cluster, ascending splits) and the final
// store scales row t by rs[t] = 1 / sqrt(sum_k x[t,k]^2 / K + eps), all IEEE operations.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace w8a8 {

constexpr int kQ8MaxWarps = 16;
constexpr int kQ8MaxBlocksPerWarp = 8;
constexpr int kQ8TargetBlocksPerWarp = 4;
// float4 per (tile, split) record of a split read: 32 lanes' partial sums, then the 8 rows' sums
// of squares (RMS-norm variant).
constexpr int kQ8Rec = 34;
// One CTA covers up to 16 warps x 8 blocks = 4096 k of a tile, so K <= 4096 needs no cross-CTA
// combine: its two dependent global round trips (counter, then the partials) cost more than the
// extra loads each warp keeps in flight.

struct Q8Params {
  const uint16_t* x;
  const uint16_t* gamma;   // RMS-norm variant: the norm weight g [K] (bf16)
  float eps;
  const int8_t* q;
  const uint16_t* d;
  uint16_t* y;
  uint32_t* status;
  uint32_t* counters;
  float4* partials;
  int T, K, N, KB, warps, splits;
  int cluster;      // > 1: CTA r of a tile's cluster runs the tile's warps r * warps .. r * warps + warps - 1
  int pdl;          // W8A8_FLAG_PDL: the weights may be read before the dependency wait
  int tile_warps;   // warps of a tile in all (the k-block runs)
};

// Two signed int8 (bytes i0, i1 of v) -> bf16x2 (i0 in the low half), exact.  In offset binary
// u = v ^ 0x80808080 each byte b sits in the float 2^23 + b (pattern 0x4B0000bb); subtracting
// 2^23 + 128 leaves the int8 value, and values in [-128, 127] are exact in bf16.
__device__ __forceinline__ uint32_t s8x2_to_bf16x2(uint32_t u, int i0, int i1) {
  const float f0 = __int_as_float((int)__byte_perm(u, 0x4B000000u, 0x7440 + i0)) - 8388736.0f;
  const float f1 = __int_as_float((int)__byte_perm(u, 0x4B000000u, 0x7440 + i1)) - 8388736.0f;
  __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 32-bit store into another CTA's shared memory (shared::cluster address).
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// rs = 1 / sqrt(ss / K + eps), each step one IEEE operation.
__device__ __forceinline__ float inv_rms(float ss, int K, float eps) {
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)K), eps)));
}

__device__ __forceinline__ void q8_store(const Q8Params& p, const float (&v)[4], int n_a, int c) {
  const int n_b = n_a + 8;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = 2 * c + (r & 1);
    const int n = (r < 2) ? n_a : n_b;
    if (t < p.T && n < p.N) p.y[(long long)t * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v[r]));
  }
}

template <bool kRms>
__global__ void __launch_bounds__(32 * kQ8MaxWarps) q8_0_gemv_kernel(const __grid_constant__ Q8Params p) {
  __shared__ float4 red[kQ8MaxWarps][32];
  __shared__ float ssred[kQ8MaxWarps][8];   // RMS-norm variant: each warp's sums of squares per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int rank = p.cluster > 1 ? (int)cluster_ctarank() : 0;
  const int tile = blockIdx.x / (p.splits * p.cluster);
  const int split = (blockIdx.x / p.cluster) % p.splits;
  const int cb0 = even_lo(split, p.KB, p.splits);
  const int cb1 = even_lo(split + 1, p.KB, p.splits);
  // This warp's run of k blocks: the tile's warps split the split's blocks into equal runs, and a
  // cluster spreads them over its CTAs (a warp past the tile's count has none).
  const int tw = rank * p.warps + warp;
  const int wb0 = cb0 + even_lo(min(tw, p.tile_warps), cb1 - cb0, p.tile_warps);
  const int wb1 = cb0 + even_lo(min(tw + 1, p.tile_warps), cb1 - cb0, p.tile_warps);
  const int nb = wb1 - wb0;
  const int n_a = tile * 16 + g, n_b = n_a + 8;

  pdl_trigger();
  // Every launch is a programmatic dependent of the work before it (q8_launch): without
  // W8A8_FLAG_PDL nothing global is read before the dependency wait, after which the previous
  // kernel's writes are visible.  Only this warp's quants and scales are prefetched into L2 first
  // (a prefetch changes no value that a later read returns), so that the loads after the wait
  // hit in L2: lane r < 16 the quants of row tile * 16 + r, lane 16 + r that row's scales.
  if (!p.pdl) {
    const int r = lane & 15;
    const long long n = (long long)tile * 16 + r;
    if (nb > 0 && n < p.N) {
      if (lane < 16) {
        bulk_prefetch_l2(p.q + n * p.K + (long long)wb0 * 32, (uint32_t)nb * 32u);
      } else {
        prefetch_l2_line(p.d + n * p.KB + wb0);
        prefetch_l2_line(p.d + n * p.KB + wb1 - 1);
      }
    }
    pdl_wait();
  }
  // Issue every load of this warp's run first: the read is latency-bound, not bandwidth-bound.
  // With W8A8_FLAG_PDL the quants and scales, weights that nothing in flight writes (the caller's
  // promise), are requested before the dependency wait; the activations after it.
  uint2 qa[kQ8MaxBlocksPerWarp], qb[kQ8MaxBlocksPerWarp];
  uint4 xv[kQ8MaxBlocksPerWarp], gv[kQ8MaxBlocksPerWarp];
  uint16_t da[kQ8MaxBlocksPerWarp], db[kQ8MaxBlocksPerWarp];
#pragma unroll
  for (int i = 0; i < kQ8MaxBlocksPerWarp; ++i) {
    qa[i] = make_uint2(0u, 0u);
    qb[i] = make_uint2(0u, 0u);
    da[i] = 0;
    db[i] = 0;
    if (i < nb) {
      const int kb = wb0 + i;
      const long long k = (long long)kb * 32 + 8 * c;
      if (n_a < p.N) {
        qa[i] = __ldg(reinterpret_cast<const uint2*>(p.q + (long long)n_a * p.K + k));
        da[i] = __ldg(p.d + (long long)n_a * p.KB + kb);
      }
      if (n_b < p.N) {
        qb[i] = __ldg(reinterpret_cast<const uint2*>(p.q + (long long)n_b * p.K + k));
        db[i] = __ldg(p.d + (long long)n_b * p.KB + kb);
      }
    }
    // The norm weight is a weight too: fetched before the dependency wait.
    if (kRms) gv[i] = i < nb ? __ldg(reinterpret_cast<const uint4*>(p.gamma + (long long)(wb0 + i) * 32 + 8 * c))
                             : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_wait();
#pragma unroll
  for (int i = 0; i < kQ8MaxBlocksPerWarp; ++i) {
    xv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (i < nb && g < p.T)
      xv[i] = __ldcg(reinterpret_cast<const uint4*>(p.x + (long long)g * p.K + (long long)(wb0 + i) * 32 + 8 * c));
  }
  // RMS-norm variant: this lane's sum of x^2 (blocks ascending, elements in order; each square is
  // exact in fp32) and its activations times g, rounded once to bf16.  The four lanes of a row
  // then add their sums (same bits in all four).
  float ss = 0.f;
  if (kRms) {
#pragma unroll
    for (int i = 0; i < kQ8MaxBlocksPerWarp; ++i) {
      if (i < nb) {
        const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
        const uint32_t gw[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = __uint_as_float(xw[e] << 16), x1 = __uint_as_float(xw[e] & 0xFFFF0000u);
          const float g0 = __uint_as_float(gw[e] << 16), g1 = __uint_as_float(gw[e] & 0xFFFF0000u);
          ss = __fadd_rn(ss, __fmul_rn(x0, x0));
          ss = __fadd_rn(ss, __fmul_rn(x1, x1));
          __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(x0, g0), __fmul_rn(x1, g1));
          o[e] = *reinterpret_cast<uint32_t*>(&h);
        }
        xv[i] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 1));
    ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 2));
  }

  // One independent 16x8 block product per 32-k block (two k16 MMAs each, all step-0 MMAs issued
  // before the step-1 ones), then the fp16 block scales applied in ascending k.
  float blk[kQ8MaxBlocksPerWarp][4];
  uint32_t af[kQ8MaxBlocksPerWarp][2][4];
#pragma unroll
  for (int i = 0; i < kQ8MaxBlocksPerWarp; ++i) {
    blk[i][0] = blk[i][1] = blk[i][2] = blk[i][3] = 0.f;
    const uint32_t ua0 = qa[i].x ^ 0x80808080u, ua1 = qa[i].y ^ 0x80808080u;
    const uint32_t ub0 = qb[i].x ^ 0x80808080u, ub1 = qb[i].y ^ 0x80808080u;
    // k 8c+0..3 (slots 2c,2c+1 <- k 8c,8c+1; slots 2c+8,2c+9 <- k 8c+2,8c+3), then k 8c+4..7
    af[i][0][0] = s8x2_to_bf16x2(ua0, 0, 1);
    af[i][0][1] = s8x2_to_bf16x2(ub0, 0, 1);
    af[i][0][2] = s8x2_to_bf16x2(ua0, 2, 3);
    af[i][0][3] = s8x2_to_bf16x2(ub0, 2, 3);
    af[i][1][0] = s8x2_to_bf16x2(ua1, 0, 1);
    af[i][1][1] = s8x2_to_bf16x2(ub1, 0, 1);
    af[i][1][2] = s8x2_to_bf16x2(ua1, 2, 3);
    af[i][1][3] = s8x2_to_bf16x2(ub1, 2, 3);
  }
#pragma unroll
  for (int st = 0; st < 2; ++st)
#pragma unroll
    for (int i = 0; i < kQ8MaxBlocksPerWarp; ++i)
      if (i < nb)
        mma_bf16_16816(blk[i], af[i][st][0], af[i][st][1], af[i][st][2], af[i][st][3], st ? xv[i].z : xv[i].x,
                       st ? xv[i].w : xv[i].y);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kQ8MaxBlocksPerWarp; ++i) {
    if (i < nb) {
      const float sa = __half2float(__ushort_as_half(da[i]));
      const float sb = __half2float(__ushort_as_half(db[i]));
      acc[0] = fmaf(sa, blk[i][0], acc[0]);
      acc[1] = fmaf(sa, blk[i][1], acc[1]);
      acc[2] = fmaf(sb, blk[i][2], acc[2]);
      acc[3] = fmaf(sb, blk[i][3], acc[3]);
    }
  }

  if (p.cluster > 1) {
    // The tile's warp partials gather in CTA 0 of the cluster (distributed shared memory), which
    // sums them in warp order, exactly as one CTA holding all the tile's warps would.
    if (tw < p.tile_warps) {
      st_cluster_v4f(cluster_map(smem_addr(&red[tw][lane]), 0u), make_float4(acc[0], acc[1], acc[2], acc[3]));
      if (kRms && c == 0) st_cluster_f32(cluster_map(smem_addr(&ssred[tw][g]), 0u), ss);
    }
    cluster_sync_all();
    if (rank != 0 || warp != 0) return;
  } else {
    red[warp][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if (kRms && c == 0) ssred[warp][g] = ss;
    __syncthreads();
    if (warp != 0) return;
  }
  // This lane stores rows t = 2c and 2c + 1: their sums of squares, in warp order too.
  float tot[4] = {0.f, 0.f, 0.f, 0.f};
  float ts0 = 0.f, ts1 = 0.f;
  for (int w = 0; w < p.tile_warps; ++w) {
    const float4 v = red[w][lane];
    tot[0] += v.x;
    tot[1] += v.y;
    tot[2] += v.z;
    tot[3] += v.w;
    if (kRms) {
      ts0 = __fadd_rn(ts0, ssred[w][2 * c]);
      ts1 = __fadd_rn(ts1, ssred[w][2 * c + 1]);
    }
  }
  if (p.splits == 1) {
    if (kRms) {
      const float r0 = inv_rms(ts0, p.K, p.eps), r1 = inv_rms(ts1, p.K, p.eps);
      tot[0] = __fmul_rn(tot[0], r0);
      tot[1] = __fmul_rn(tot[1], r1);
      tot[2] = __fmul_rn(tot[2], r0);
      tot[3] = __fmul_rn(tot[3], r1);
    }
    q8_store(p, tot, n_a, c);
    return;
  }
  float4* mine = p.partials + ((long long)tile * p.splits + split) * kQ8Rec;
  __stcg(mine + lane, make_float4(tot[0], tot[1], tot[2], tot[3]));
  if (kRms && lane < 4) __stcg(reinterpret_cast<float2*>(mine + 32) + lane, make_float2(ts0, ts1));
  __threadfence();
  __syncwarp();
  uint32_t old = 0;
  if (lane == 0) old = atomicAdd(p.counters + tile, 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old >= (uint32_t)p.splits) {
    if (lane == 0) atomicOr(p.status, W8A8_DEV_COUNTER_CORRUPT);
    return;
  }
  if (old != (uint32_t)p.splits - 1) return;
  __threadfence();
  // Ascending split order; each batch's loads are all in flight before the first is used.
  float sum[4] = {0.f, 0.f, 0.f, 0.f};
  float ssum0 = 0.f, ssum1 = 0.f;
  for (int base = 0; base < p.splits; base += 8) {
    float4 v[8];
    float2 sv[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int s = base + b;
      v[b] = make_float4(tot[0], tot[1], tot[2], tot[3]);
      sv[b] = make_float2(ts0, ts1);
      if (s < p.splits && s != split) {
        const float4* rec = p.partials + ((long long)tile * p.splits + s) * kQ8Rec;
        v[b] = __ldcg(rec + lane);
        if (kRms) sv[b] = __ldcg(reinterpret_cast<const float2*>(rec + 32) + c);
      }
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (base + b < p.splits) {
        sum[0] += v[b].x;
        sum[1] += v[b].y;
        sum[2] += v[b].z;
        sum[3] += v[b].w;
        if (kRms) {
          ssum0 = __fadd_rn(ssum0, sv[b].x);
          ssum1 = __fadd_rn(ssum1, sv[b].y);
        }
      }
    }
  }
  if (lane == 0) atomicExch(p.counters + tile, 0u);
  if (kRms) {
    const float r0 = inv_rms(ssum0, p.K, p.eps), r1 = inv_rms(ssum1, p.K, p.eps);
    sum[0] = __fmul_rn(sum[0], r0);
    sum[1] = __fmul_rn(sum[1], r1);
    sum[2] = __fmul_rn(sum[2], r0);
    sum[3] = __fmul_rn(sum[3], r1);
  }
  q8_store(p, sum, n_a, c);
}

int q8_plan(int T, int K, int N, Q8Plan* plan) {
  if (T < 1 || T > 8 || K < 1 || K > 65536 || N < 1 || N > 1048576) return W8A8_ERR_INVALID_ARG;
  if (K % 32 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
  Q8Plan pl{};
  pl.n_tiles = (N + 15) / 16;
  pl.kb = K / 32;
  const int per_cta_max = kQ8MaxWarps * kQ8MaxBlocksPerWarp;
  pl.splits = (pl.kb + per_cta_max - 1) / per_cta_max;
  const int per_split = (pl.kb + pl.splits - 1) / pl.splits;
  const int warps = (per_split + kQ8TargetBlocksPerWarp - 1) / kQ8TargetBlocksPerWarp;
  pl.warps = warps < kQ8MaxWarps ? warps : kQ8MaxWarps;   // then at most 8 blocks per warp
  // A tile read by one CTA with four or more warps spreads its warps over a cluster, two per CTA:
  // more SMs pull the weight, the partials meet in distributed shared memory in the same order,
  // and the sums are bit-identical to the one-CTA read.
  pl.tile_warps = pl.warps;
  pl.cluster = 1;
  if (pl.splits == 1 && pl.warps >= 4) {
    pl.cluster = (pl.warps + 1) / 2;
    pl.warps = 2;
  }
  pl.blocks = pl.n_tiles * pl.splits * pl.cluster;
  const size_t counters = ((size_t)pl.n_tiles * 4 + 255) / 256 * 256;
  const size_t partials = pl.splits > 1 ? (size_t)pl.n_tiles * pl.splits * kQ8Rec * 16 : 0;
  pl.counters_offset = kWsHeaderBytes;
  pl.partials_offset = kWsHeaderBytes + counters;
  pl.workspace_bytes = kWsHeaderBytes + counters + partials;
  *plan = pl;
  return W8A8_OK;
}

cudaError_t q8_launch(const Q8Plan& pl, const void* x, const int8_t* q, const void* d, void* y, int T, int K, int N,
                      void* ws, bool pdl, cudaStream_t stream, const void* gamma, float eps) {
  Q8Params p;
  p.x = static_cast<const uint16_t*>(x);
  p.gamma = static_cast<const uint16_t*>(gamma);
  p.eps = eps;
  p.q = q;
  p.d = static_cast<const uint16_t*>(d);
  p.y = static_cast<uint16_t*>(y);
  p.status = static_cast<uint32_t*>(ws);
  p.counters = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + pl.counters_offset);
  p.partials = reinterpret_cast<float4*>(static_cast<uint8_t*>(ws) + pl.partials_offset);
  p.T = T;
  p.K = K;
  p.N = N;
  p.KB = pl.kb;
  p.warps = pl.warps;
  p.splits = pl.splits;
  p.cluster = pl.cluster;
  p.tile_warps = pl.tile_warps;
  p.pdl = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.blocks);
  cfg.blockDim = dim3((unsigned)(32 * pl.warps));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // Always a programmatic dependent of the work before it (see the kernel: without the flag nothing
  // global is touched before the dependency wait).
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (pl.cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)pl.cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = gamma ? cudaLaunchKernelEx(&cfg, q8_0_gemv_kernel<true>, p) : cudaLaunchKernelEx(&cfg, q8_0_gemv_kernel<false>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace w8a8
