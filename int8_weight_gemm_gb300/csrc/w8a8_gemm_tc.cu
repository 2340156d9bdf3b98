// W8A8 GEMM for 32 < M <= 128 on the fifth-generation tensor cores (tcgen05, sm_103a):
// out[M,N] = bf16((float(x_q @ W) * x_scale) * w_scale), the same operator and the same packed
// weight as the decode kernel.
//
// Operator: "INT8 W8A8 GEMM - Decode (M <= 32) - gfx928 / SGLang TP4", header paragraph.  Its
// section 3 ("Boundary: 16 < M <= 32") keeps a staged arm for larger M next to the decode arm, for
// the same (K, N): the decode pattern does not carry over once M grows.  This file is that arm.
// Split-K and the last-arrival combine follow the page's section 1.1 (qkv recipe): monotonic
// work split over the SM count, per-tile arrival counters in the workspace, the last arriver sums
// the partials, scales them and stores bf16, and every call leaves the counters and sums zeroed.
//
// Why tcgen05 here.  With M activation rows, every weight byte feeds 2M multiply-adds; at M = 128
// a weight stream at HBM speed needs ~1.8 PFLOP/s, three times what the register-fed mma.sync path
// of this part sustains, so the multiply moves to tcgen05.mma (M = 128 weight rows, N = 64 or 128
// activation rows, K = 16, f32 accumulation in tensor memory).  int8 tensor MMAs do not exist on
// sm_103a (ptxas rejects kind::i8), so every int8 is converted exactly to fp16 (each int8 value
// is an fp16 integer) and multiplied with kind::f16.
//
// Exactness.  A product is an integer of magnitude <= 2^14; one accumulator collects at most
// 512 k (four stages) before it is read out, so every f32 accumulator value is an integer of
// magnitude <= 2^23 and exact.  The read-out converts it to int32 (exact) and adds it to int32
// sums; split tiles add int32 partials.  The result is the int32 sum an int8 MMA would give, bit
// for bit, whatever the split.
//
// One call is two launches:
//  * x16: the activations converted once to fp16 (exact) into the workspace, in the k order the
//    converted weight has in tensor memory, so that no CTA converts them again; it lets the GEMM
//    launch at once (programmatic dependent launch);
//  * the GEMM (one CTA per SM, all of its tensor memory), launched as a programmatic dependent of
//    x16: its weight stream starts while x16 runs.  Roles:
//    - weight producer (one thread): per stage of 128 k, two 1-D bulk copies of packed weight (the
//      CTA's 128-row tile is two consecutive 64-row packed tiles) into a deep ring that the
//      converter warps free as soon as they have read a stage, so it holds the bytes in flight
//      from HBM;
//    - activation producer (one thread): per stage two 2-D tensor-map boxes of fp16 activations
//      (64 k x N_mma rows each, 128-byte swizzle: the MMA's B operand as it lands) into a short
//      ring that the MMAs free;
//    - sixteen converter warps in four groups: group g writes the weight rows of every stage
//      q with q % 4 == g into tensor-memory A slot g as the fp16 A operand (tcgen05.st, lane =
//      row, one packed 16-byte chunk per thread and store), so four stages convert at once.  All
//      sixteen read the accumulators out at the end of each period (512 k), once its MMAs have
//      completed, and keep int32 sums in registers (each warp one lane quarter and one quarter of
//      the columns); at the end of a segment they store bf16 or add the split tile's partial and,
//      as the last arrival, finish it;
//    - one or two MMA-issuing threads (two take alternate k-steps into their own accumulators);
//      a period's last MMAs signal the read-out, and the read-out frees the accumulator buffer.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace w8a8 {
namespace tc {

constexpr int kPackRows = 64;                        // rows of a packed tile
constexpr int kTileRows = 128;                       // weight rows of a CTA tile = MMA M
constexpr int kKBlock = 32;                          // k per unit of the split
constexpr int kPackSlab = kPackRows * kKBlock;       // 2048: one packed slab
constexpr int kStageUnits = 4;                       // 32-k units per stage
constexpr int kStageK = kStageUnits * kKBlock;       // 128
constexpr int kBoxK = 64;                            // k of one activation box (128 bytes of fp16)
constexpr int kHalfBytes = kStageUnits * kPackSlab;  // one packed tile's share of a stage: 8 KiB
constexpr int kWStage = 2 * kHalfBytes;              // 16 KiB of weight per stage
constexpr int kConvWarps = 16;                       // four per tensor-memory lane quarter
constexpr int kConvThreads = 32 * kConvWarps;
// The converter warps form four groups of four (one warp per lane quarter each); group g converts
// every stage q with q % 4 == g, whole, into tensor-memory A slot g.  Four stages are then
// converted at once, and a warp meets the pipeline's barriers once per four stages.
constexpr int kConvGroups = 4;
constexpr int kGroupWarps = kConvWarps / kConvGroups;
constexpr int kWProducerWarp = kConvWarps;           // streams the packed weight
constexpr int kBProducerWarp = kConvWarps + 1;       // loads the activation boxes
constexpr int kMmaWarp = kConvWarps + 2;             // first MMA-issuing warp; owns tensor memory
constexpr int kPeriodStages = 4;                     // stages per accumulator read-out (512 k)
constexpr int kTmemCols = 512;
constexpr int kACols = kStageK / 2;                  // tensor-memory columns of one A stage (fp16 pairs)
constexpr int kConvBarrier = 1;                      // named barrier of the converter warps

template <int NT16>
struct TcLayout {
  static constexpr int kN = 16 * NT16;               // MMA N: activation rows (zero past M)
  // The issue cost of an MMA is per instruction, so the widest MMA (N = kN) is the cheapest.  At
  // N = 64 two threads issue, each every other k-step of a stage into its own accumulators (the
  // read-out adds them); at N = 128 the accumulators of a second thread would not fit next to the A
  // ring, and one thread issues.  (Splitting the activation rows between two threads instead gives
  // each the same number of MMAs and was measured to gain nothing.)
  static constexpr int kIssuers = kN <= 64 ? 2 : 1;
  // The weight ring is freed as soon as the converter warps have read a stage, so it can be deep:
  // it holds the bytes in flight from HBM.  The activation ring (from L2) is freed by the MMAs.
  static constexpr int kWStages = kN <= 64 ? 10 : 8;
  static constexpr int kBStages = kN <= 64 ? 4 : 3;
  static constexpr int kOpStages = kConvGroups;       // tensor-memory A slots: one per converter group
  static constexpr int kBBox = kN * 128;              // one fp16 activation box (1 KiB multiple)
  static constexpr int kBStage = 2 * kBBox;
  static constexpr int kDCol0 = kOpStages * kACols;   // first accumulator column
  static constexpr int kThreads = 32 * (kMmaWarp + kIssuers);
  static constexpr int kBytes = 1024 + kBStages * kBStage + kWStages * kWStage;   // boxes first: 1 KiB aligned
  static constexpr int kCols = kN / 4;                // accumulator columns per converter warp
  static_assert(kDCol0 + kIssuers * 2 * kN <= kTmemCols, "tensor-memory columns");
  static_assert(kBytes <= 232448 - 2048, "shared memory");
};

struct TcParams {
  CUtensorMap xmap;     // fp16 activations [M,K] in the workspace, box 64 x N_mma, 128-byte swizzle
  const uint8_t* wp;    // packed weight (64-row tiles of 2 KiB slabs)
  const float* x_scale;
  const float* w_scale;
  uint16_t* out;
  uint32_t* status;
  uint32_t* counters;   // [tile] arrivals at a split tile, zero between calls
  int* planes;          // [tile][m < N_mma][row < 128] int32 sums of a split tile, zero between calls
  GemmSplit split;      // over the 128-row tiles, in 32-k units
  int M, N, KB, tiles64;
  int* acc_out;         // optional: the exact int32 sums [M, N] row-major, stored beside out
  int debug_stall;      // test hook: one converter warp of CTA 0 waits on a barrier that nothing completes
};

// The CTA's schedule: its run of units [b0, b1) is a sequence of segments (one tile's part each),
// a segment is a sequence of stages of at most kStageUnits units, and consecutive stages of a
// segment form accumulation periods of at most kPeriodStages.  Every role walks the same sequence.
struct Walk {
  int u, b1, KB, t, seg_begin, seg_end, ns, q, sp, period;
  __device__ Walk(int b0, int b1_, int KB_) : u(b0), b1(b1_), KB(KB_), q(0), sp(0), period(0) { begin_segment(); }
  __device__ void begin_segment() {
    t = u / KB;
    seg_begin = u;
    seg_end = min(b1, (t + 1) * KB);
    ns = min(kStageUnits, seg_end - u);
  }
  __device__ bool done() const { return u >= b1; }
  __device__ bool seg_first() const { return u == seg_begin; }
  __device__ bool seg_last() const { return u + ns >= seg_end; }
  __device__ bool period_first() const { return sp == 0; }
  __device__ bool period_last() const { return seg_last() || sp == kPeriodStages - 1; }
  __device__ bool whole_tile() const { return seg_begin == t * KB && seg_end == (t + 1) * KB; }
  __device__ int kb0() const { return u - t * KB; }
  __device__ void next() {
    const bool pl = period_last(), sl = seg_last();
    u += ns;
    ++q;
    if (pl) {
      sp = 0;
      ++period;
    } else {
      ++sp;
    }
    if (u >= b1) return;
    if (sl) begin_segment();
    else ns = min(kStageUnits, seg_end - u);
  }
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// 8 consecutive tensor-memory columns of this thread's lane (warp-wide).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}

// Shared-memory matrix descriptor, K-major with the 128-byte swizzle: rows of 128 bytes (64 fp16
// of k), 16-byte chunks XOR-ed with the row index mod 8, atoms of 8 rows 1024 bytes apart (the
// stride field), the leading-dimension field unused (1).  Layout type 2 in bits 61..63, descriptor
// version 1 in bits 46..47, base offset 0 (atoms 1024-byte aligned).  Within an atom the k-steps
// of 16 start 32 bytes apart: the swizzle applies to the address bits, so the start moves by the
// unswizzled offset.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// int32 load that bypasses L1 (the partial sums of other CTAs).
__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One output element: bf16_rne((float(acc) * x_scale[m]) * w_scale[n]).
__device__ __forceinline__ uint16_t epilogue(int acc, float xsv, float wsv) {
  float f = __int2float_rn(acc);
  f = __fmul_rn(f, xsv);
  f = __fmul_rn(f, wsv);
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Bounded wait for the phase of `parity`: mbar_wait (one non-blocking test, then suspended
// try_wait polls that leave the issue slots to the working warps).  With converter groups (each
// warp meets the pipeline's barriers once per four stages) suspended waits measured faster than
// polling with short sleeps (gate_up-sized M = 64 58.0 -> 55.0 us, M = 128 70.6 -> 68.2 us); with
// every warp converting every stage they had measured slower.  Gives up when another thread has
// raised *abort, or after `limit` cycles (then records the timeout in *status and raises *abort).
// Returns true when the phase completed.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status,
                                        long long limit = kWaitTimeoutCycles) {
  return mbar_wait(bar, parity, abort, status, limit);
}

// tc_wait taken by a whole warp: the warp goes on only if every lane saw the phase complete, so
// the warp-wide tensor-memory instructions after it always run with all 32 lanes.
__device__ __forceinline__ bool mbar_wait_all(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status) {
  const bool ok = tc_wait(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Bounded wait on one phase of `bar` for a whole warp: lane 0 polls, the other lanes wait for it at
// the warp barrier of the broadcast; the outcome is the same for all 32 lanes.  For waits whose next
// step is a tensor-memory instruction behind tcgen05.fence::after_thread_sync.
__device__ __forceinline__ bool mbar_wait_lane0(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status,
                                                long long limit = kWaitTimeoutCycles) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = tc_wait(bar, parity, abort, status, limit) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// One arrival for the warp, after every lane's earlier work (the warp barrier orders it): the
// barriers the converter warps signal count warps, not threads.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Bounded meeting of all converter warps on one phase of `bar` (count kConvWarps).
__device__ __forceinline__ bool conv_sync(uint64_t* bar, uint32_t& phase, volatile int* abort, uint32_t* status) {
  mbar_arrive_warp(bar);
  const bool ok = mbar_wait_lane0(bar, phase, abort, status);
  phase ^= 1u;
  return ok;
}

// The weight's k order inside tensor memory.  A converter thread writes one packed 16-byte chunk
// (rows g and g + 8 of a 16-row group, k = 8c ... 8c + 7 of a 32-k unit) with the 16x256b shape, so
// tensor-memory column j of the unit (the MMA's k pair 2j, 2j + 1) holds the weight pair
// k = 8 ((j % 8) / 2) + 2 ((j % 2) + 2 (j / 8)) + {0, 1}.  In groups of four k: the MMA's groups
// 0 ... 7 of a unit are the weight's groups 0, 2, 4, 6, 1, 3, 5, 7.  The activations are written in
// the same order, so every product pairs the same k on both sides and the dot product is the
// plain sum over k.

// int8 activations -> fp16 (exact) in the MMA's k order, one 32-k unit of one row per thread step.
__global__ void __launch_bounds__(256) x16_kernel(const uint4* __restrict__ x, uint4* __restrict__ x16, long long units) {
  pdl_trigger();   // the GEMM may launch now: it streams weight until this grid has completed
  pdl_wait();      // x_q may come from the previous grid, and the previous call may still read x16
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < units; i += stride) {
    const uint4 a = __ldg(x + 2 * i), b = __ldg(x + 2 * i + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t h[16];   // group gi of four k as fp16 pairs h[2 gi], h[2 gi + 1]
#pragma unroll
    for (int gi = 0; gi < 8; ++gi) offset_bytes_to_half2_pairs(w[gi] ^ 0x80808080u, h[2 * gi], h[2 * gi + 1]);
    uint4* o = x16 + 4 * i;
    o[0] = make_uint4(h[0], h[1], h[4], h[5]);      // groups 0, 2
    o[1] = make_uint4(h[8], h[9], h[12], h[13]);    // groups 4, 6
    o[2] = make_uint4(h[2], h[3], h[6], h[7]);      // groups 1, 3
    o[3] = make_uint4(h[10], h[11], h[14], h[15]);  // groups 5, 7
  }
}

// 16 lanes x 16 columns: thread t writes lanes t / 4 (v0, v1, v4, v5) and t / 4 + 8 (v2, v3, v6, v7),
// columns 2 (t % 4), 2 (t % 4) + 1 (v0 ... v3) and the same plus 8 (v4 ... v7); warp-wide.
__device__ __forceinline__ void tmem_st_16x256_x2(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x2.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

template <int NT16>
__global__ void __launch_bounds__(TcLayout<NT16>::kThreads, 1) w8a8_gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using L = TcLayout<NT16>;
  constexpr int kN = L::kN;
  constexpr int kI = L::kIssuers;
  constexpr int NW = L::kWStages;
  constexpr int NB = L::kBStages;
  constexpr int NA = L::kOpStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t wfull_bar[NW];   // a weight stage landed
  __shared__ __align__(8) uint64_t wempty_bar[NW];  // the converter warps have read a weight stage
  __shared__ __align__(8) uint64_t bfull_bar[NB];   // an activation stage (two boxes) landed
  __shared__ __align__(8) uint64_t bdone_bar[NB];   // the MMAs reading an activation stage completed
  __shared__ __align__(8) uint64_t adone_bar[NA];   // the MMAs reading a tensor-memory A stage completed
  __shared__ __align__(8) uint64_t conv_bar[NA];    // a tensor-memory A stage written by its converter group
  __shared__ __align__(8) uint64_t dfull_bar[2];    // the MMAs of an accumulation period completed
  __shared__ __align__(8) uint64_t dempty_bar[2];   // an accumulator buffer has been read out
  __shared__ __align__(8) uint64_t final_bar[kI];   // every MMA of an issuer completed
  __shared__ __align__(8) uint64_t sync_bar;        // converter warps meet at a split tile's combine
  __shared__ __align__(8) uint64_t stall_bar;       // test hook only: never completed
  __shared__ uint32_t tmem_base;
  __shared__ float xs_sm[kN];
  __shared__ int abort_flag;
  __shared__ uint32_t last_flag;

  // NB x [activation box k 0..63 | box k 64..127] (1 KiB aligned for the swizzle), then NW weight stages.
  uint8_t* const bring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* const wring = bring + NB * L::kBStage;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NW; ++s) {
      mbar_init(&wfull_bar[s], 1);
      mbar_init(&wempty_bar[s], kGroupWarps);
    }
#pragma unroll
    for (int s = 0; s < NB; ++s) {
      mbar_init(&bfull_bar[s], 1);
      mbar_init(&bdone_bar[s], kI);
    }
#pragma unroll
    for (int a = 0; a < NA; ++a) {
      mbar_init(&adone_bar[a], kI);
      mbar_init(&conv_bar[a], kGroupWarps);
    }
#pragma unroll
    for (int d = 0; d < 2; ++d) {
      mbar_init(&dfull_bar[d], kI);
      mbar_init(&dempty_bar[d], kConvWarps);
    }
#pragma unroll
    for (int i = 0; i < kI; ++i) mbar_init(&final_bar[i], 1);
    mbar_init(&sync_bar, kConvWarps);
    mbar_init(&stall_bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();   // the next call on the stream may start its own launches
  const uint32_t tmem = tmem_base;

  int b0, b1;
  gemm_split_run(p.split, blockIdx.x, &b0, &b1);

  if (warp == kWProducerWarp) {
    // ---------------------------------------------------------------- weight producer (one thread)
    // The packed weight is never written by the work this grid depends on, so this thread never
    // waits for it: the weight streams from the first cycle.
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      int q = 0;
      for (Walk it(b0, b1, p.KB); !it.done(); it.next(), ++q) {
        const int s = q % NW;
        if (q >= NW && !tc_wait(&wempty_bar[s], (uint32_t)(((q / NW) & 1) ^ 1), &abort_flag, p.status)) break;
        const int t64 = 2 * it.t;
        const bool two = t64 + 1 < p.tiles64;
        const uint32_t bytes = (uint32_t)(it.ns * kPackSlab);
        mbar_arrive_expect_tx(&wfull_bar[s], bytes * (two ? 2u : 1u));
        uint8_t* dst = wring + s * kWStage;
        const uint8_t* src = p.wp + ((size_t)t64 * p.KB + it.kb0()) * kPackSlab;
        bulk_g2s_hint(dst, src, bytes, &wfull_bar[s], policy);
        if (two) bulk_g2s_hint(dst + kHalfBytes, src + (size_t)p.KB * kPackSlab, bytes, &wfull_bar[s], policy);
      }
      // Every copy issued must land before the CTA may exit.
      for (int s = 0; s < NW && s < q; ++s) {
        const int last = s + NW * ((q - 1 - s) / NW);
        mbar_wait_drain(&wfull_bar[s], (uint32_t)((last / NW) & 1), p.status);
      }
    }
  } else if (warp == kBProducerWarp) {
    // ---------------------------------------------------------------- activation producer (one thread)
    if (lane == 0) {
      tma_prefetch_desc(&p.xmap);
      pdl_wait();   // the fp16 activations are written by the grid this one depends on
      int q = 0;
      for (Walk it(b0, b1, p.KB); !it.done(); it.next(), ++q) {
        const int s = q % NB;
        // The slot is free once the MMAs of stage q - NB (which read it) have completed.
        if (q >= NB && !tc_wait(&bdone_bar[s], (uint32_t)(((q - NB) / NB) & 1), &abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&bfull_bar[s], (uint32_t)L::kBStage);
        const int k0 = it.kb0() * kKBlock;
        tma_load_2d(bring + s * L::kBStage, &p.xmap, k0, 0, &bfull_bar[s]);
        tma_load_2d(bring + s * L::kBStage + L::kBBox, &p.xmap, k0 + kBoxK, 0, &bfull_bar[s]);
      }
      for (int s = 0; s < NB && s < q; ++s) {
        const int last = s + NB * ((q - 1 - s) / NB);
        mbar_wait_drain(&bfull_bar[s], (uint32_t)((last / NB) & 1), p.status);
      }
    }
  } else if (warp >= kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuers (one thread each)
    const int issuer = warp - kMmaWarp;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kTileRows, kN);
      bool started = false;   // this issuer's accumulator of the current period holds a k-step
      for (Walk it(b0, b1, p.KB); !it.done(); it.next()) {
        const int sb = it.q % NB;
        const int a = it.q % NA;
        const int db = it.period & 1;
        if (it.period_first() && it.period >= 2 &&
            !tc_wait(&dempty_bar[db], (uint32_t)(((it.period >> 1) - 1) & 1), &abort_flag, p.status))
          break;
        // Both operands: the A slot written by its converter group, the activation stage landed.
        if (!tc_wait(&conv_bar[a], (uint32_t)((it.q / NA) & 1), &abort_flag, p.status)) break;
        if (!tc_wait(&bfull_bar[sb], (uint32_t)((it.q / NB) & 1), &abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_addr = tmem + (uint32_t)(L::kDCol0 + (issuer * 2 + db) * kN);
        const uint32_t a_addr = tmem + (uint32_t)(a * kACols);
        const uint32_t b_addr = smem_addr(bring + sb * L::kBStage);
        if (it.period_first()) started = false;
        // k-step j covers k in [16 j, 16 j + 16) of the stage: A columns 8 j ... 8 j + 7; B in box
        // j / 4 at byte 32 (j % 4) of each 128-byte row.  Every issuer has at least one k-step per
        // stage (a stage has 2 ns >= 2 of them).
        for (int j = issuer; j < 2 * it.ns; j += kI) {
          const uint64_t bdesc = smem_desc_sw128(b_addr + (uint32_t)((j >> 2) * L::kBBox + (j & 3) * 32));
          umma_f16_tmem_a(d_addr, a_addr + 8u * j, bdesc, idesc, started);
          started = true;
        }
        // Each completes once these MMAs (and every earlier one of this thread) have completed: the
        // activation slot and the A stage are free again and, at a period's end, the converter warps
        // may read the accumulators.
        umma_commit(&bdone_bar[sb]);
        umma_commit(&adone_bar[a]);
        if (it.period_last()) umma_commit(&dfull_bar[db]);
      }
      // Whatever happened above, every MMA this thread issued completes before tensor memory is freed.
      umma_commit(&final_bar[issuer]);
      mbar_wait_drain(&final_bar[issuer], 0, p.status);
    }
  } else {
    // ---------------------------------------------------------------- converter warps
    // Warp w owns tensor-memory lanes 32 (w % 4) ... + 31 (rows of the CTA tile) and accumulator
    // columns (w / 4) kN / 4 ... + kN / 4 - 1, and converts its 32 rows of every stage q with
    // q % 4 == w / 4 (its group), all units of the stage, into A slot w / 4.  Its 32 rows are two
    // 16-row groups s of packed tile (w % 4) / 2; the packed 16-byte chunk (s, lane) of a unit holds
    // k = 8c ... 8c + 7 of rows g and g + 8 (g = lane / 4, c = lane % 4; words: row g k 8c.., row
    // g + 8 k 8c.., row g k 8c+4.., row g + 8 k 8c+4..), which is what the 16x256b store takes from
    // thread `lane`: one 16-byte read (a group is 512 contiguous bytes), four exact conversions, one
    // store per group and unit.  Every warp reads out every accumulation period (its columns of its
    // lanes), four stages after the period's last one.
    const int quad = warp & 3, unit = warp >> 2;   // unit: the converter group, and the column quarter
    const int half = quad >> 1;
    const int s16 = 2 * (quad & 1);
    const uint32_t t_lane = tmem + ((uint32_t)(32 * quad) << 16);
    const int row = 32 * quad + lane;
    const int m0 = unit * L::kCols;

    pdl_wait();   // x_scale, w_scale, out and the workspace may belong to earlier work on the stream
    for (int i = threadIdx.x; i < kN; i += kConvThreads) xs_sm[i] = i < p.M ? __ldg(p.x_scale + i) : 0.f;
    named_bar_sync(kConvBarrier, kConvThreads);

    int iacc[L::kCols];
#pragma unroll
    for (int c = 0; c < L::kCols; ++c) iacc[c] = 0;
    float wsv = 0.f;
    uint32_t sync_phase = 0;
    Walk dr(b0, b1, p.KB);   // the next stage to retire (its MMAs have completed)

    // Retire stage dr: at a period's end add its accumulators to the int32 sums and hand the buffer
    // back to the issuers; at a segment's end store the tile part or combine it.  False on abort.
    auto retire = [&]() -> bool {
      const int n = dr.t * kTileRows + row;
      if (dr.seg_first()) wsv = n < p.N ? __ldg(p.w_scale + n) : 0.f;
      if (dr.period_last()) {
        const int db = dr.period & 1;
        if (!mbar_wait_lane0(&dfull_bar[db], (uint32_t)((dr.period >> 1) & 1), &abort_flag, p.status)) return false;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < kI; ++i) {
#pragma unroll
          for (int c0 = 0; c0 < L::kCols; c0 += 8) {
            uint32_t d[8];
            tmem_ld8(t_lane + (uint32_t)(L::kDCol0 + (i * 2 + db) * kN + m0 + c0), d);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c) iacc[c0 + c] += __float2int_rn(__uint_as_float(d[c]));
          }
        }
        tc_fence_before();
        mbar_arrive_warp(&dempty_bar[db]);
        if (dr.seg_last()) {
          // Element (m0 + c, n) of out, walked down the column one activation row at a time.
          uint16_t* o = p.out + (size_t)m0 * p.N + n;
          const int mrows = min(L::kCols, p.M - m0);   // rows of this warp's columns that exist
          if (dr.whole_tile()) {
            if (n < p.N) {
#pragma unroll
              for (int c = 0; c < L::kCols; ++c, o += p.N)
                if (c < mrows) {
                  *o = epilogue(iacc[c], xs_sm[m0 + c], wsv);
                  if (p.acc_out) p.acc_out[(size_t)(m0 + c) * p.N + n] = iacc[c];
                }
            }
          } else {
            // Split tile: add this partial to the tile's int32 plane, count the arrival (one thread,
            // release / acquire), and let the last arrival read the total, store bf16 and zero the plane.
            int* const plane = p.planes + ((size_t)dr.t * kN + m0) * kTileRows + row;
            if (n < p.N) {
#pragma unroll
              for (int c = 0; c < L::kCols; ++c)
                if (c < mrows) red_add_s32(plane + c * kTileRows, iacc[c]);
            }
            __threadfence();
            if (!conv_sync(&sync_bar, sync_phase, &abort_flag, p.status)) return false;
            if (threadIdx.x == 0) {
              const uint32_t arrivals = (uint32_t)gemm_split_contributors(p.split, dr.t);
              const uint32_t old = atom_add_acq_rel_u32(p.counters + dr.t, 1u);
              if (old >= arrivals) atomicOr(p.status, W8A8_DEV_COUNTER_CORRUPT);
              const uint32_t last = old == arrivals - 1 ? 1u : 0u;
              if (last) p.counters[dr.t] = 0u;   // every contributor has arrived: ready for the next call
              last_flag = last;
            }
            if (!conv_sync(&sync_bar, sync_phase, &abort_flag, p.status)) return false;
            if (last_flag) {
              __threadfence();
              if (n < p.N) {
#pragma unroll 8
                for (int c = 0; c < L::kCols; ++c, o += p.N) {
                  if (c < mrows) {
                    int* const w = plane + c * kTileRows;
                    const int total = ld_relaxed_s32(w);
                    *w = 0;
                    *o = epilogue(total, xs_sm[m0 + c], wsv);
                    if (p.acc_out) p.acc_out[(size_t)(m0 + c) * p.N + n] = total;
                  }
                }
              }
            }
          }
#pragma unroll
          for (int c = 0; c < L::kCols; ++c) iacc[c] = 0;
        }
      }
      dr.next();
      return true;
    };

    bool ok = true;
    if (p.debug_stall && blockIdx.x == 0 && warp == 0) {
      // Test hook of the device fault path (after the converter warps' named barrier, which every
      // one of them must reach): this warp waits, with a short bound, on a barrier that nothing
      // completes.  The wait runs out, records W8A8_DEV_WAIT_TIMEOUT and raises the abort flag;
      // every other role gives up at its next wait, the issuers after their MMAs have completed and
      // the producers after their copies have landed, and all meet at the final barrier before the
      // tensor memory is freed.
      mbar_wait_lane0(&stall_bar, 0u, &abort_flag, p.status, kTestStallCycles);
      ok = false;
    }
    for (Walk it(b0, b1, p.KB); ok && !it.done(); it.next()) {
      // Stage q - 4 retires as the walk passes stage q: at a period's end this reads the period's
      // accumulators once its MMAs have completed.
      if (it.q >= kConvGroups && !retire()) {
        ok = false;
        break;
      }
      if ((it.q & (kConvGroups - 1)) != unit) continue;   // another group converts this stage
      const int s = it.q % NW;
      const int a = unit;   // this group's A slot
      if (!mbar_wait_all(&wfull_bar[s], (uint32_t)((it.q / NW) & 1), &abort_flag, p.status)) {
        ok = false;
        break;
      }
      // The A slot is free once the MMAs of the group's previous stage, q - 4, have completed.
      if (it.q >= kConvGroups &&
          !mbar_wait_lane0(&adone_bar[a], (uint32_t)(((it.q - kConvGroups) / NA) & 1), &abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool have = 2 * it.t + half < p.tiles64;   // this packed tile exists (warp-uniform)
      if (have) {
        const uint8_t* wsrc = wring + s * kWStage + half * kHalfBytes;
        for (int u = 0; u < it.ns; ++u) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint4 w = lds128(wsrc + u * kPackSlab + ((s16 + r) * 32 + lane) * 16);
            uint32_t h[8];
            offset_bytes_to_half2_pairs(w.x, h[0], h[1]);   // row g,     k 8c .. 8c+3
            offset_bytes_to_half2_pairs(w.y, h[2], h[3]);   // row g + 8, k 8c .. 8c+3
            offset_bytes_to_half2_pairs(w.z, h[4], h[5]);   // row g,     k 8c+4 .. 8c+7
            offset_bytes_to_half2_pairs(w.w, h[6], h[7]);   // row g + 8, k 8c+4 .. 8c+7
            tmem_st_16x256_x2(t_lane + ((uint32_t)(16 * r) << 16) + (uint32_t)(a * kACols + 16 * u), h);
          }
        }
      }
      // Every weight value of the stage has been read and used: the slot goes back to the producer.
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty_bar[s]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&conv_bar[a]);
    }
    // Retire the stages still in flight.
    while (ok && !dr.done()) {
      if (!retire()) break;
    }
  }

  // Every role ends here: the issuers have seen all their MMAs complete and the producer all its
  // copies land; then the allocating warp returns the tensor memory.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int NT16>
static cudaError_t launch_tc(const TcParams& p, int blocks, cudaStream_t stream) {
  auto kern = w8a8_gemm_tc_kernel<NT16>;
  const int smem = TcLayout<NT16>::kBytes;
  cudaError_t e = ensure_smem_attribute((const void*)kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(TcLayout<NT16>::kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  // Always a programmatic dependent of the x16 launch just before it.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static cudaError_t launch_x16(const int8_t* x, void* x16, long long units, bool pdl, cudaStream_t stream) {
  long long grid = (units + 255) / 256;
  if (grid > 8 * kDefaultSmCount) grid = 8 * kDefaultSmCount;   // grid-stride beyond a few waves
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid < 1 ? 1 : grid));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, x16_kernel, reinterpret_cast<const uint4*>(x), static_cast<uint4*>(x16), units);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tc

int tc_plan(int M, int K, int N, int blocks, int sm_count, TcPlan* plan) {
  if (M <= kDecodeMaxM || M > kTcMaxM || K < 1 || K > 65536 || N < 1 || N > 1048576 || blocks < 0)
    return W8A8_ERR_INVALID_ARG;
  if (K % 32 != 0 || N % 8 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
  TcPlan pl{};
  pl.mma_n = M <= 64 ? 64 : 128;
  pl.tiles64 = (N + tc::kPackRows - 1) / tc::kPackRows;
  pl.n_tiles = (pl.tiles64 + 1) / 2;
  pl.kb = K / tc::kKBlock;
  pl.units = (long long)pl.n_tiles * pl.kb;
  if (blocks == 0) {
    // At most one CTA per SM: each holds all of its SM's tensor memory and most of its shared
    // memory.  With at least as many tiles as SMs, a CTA count that divides the tile count gives
    // every CTA whole tiles, so no tile needs a combine; at M = 128 a tile's partial sums are as
    // large as 512 k of its weight, and such a plan was measured faster (gate_up-sized, 192
    // tiles: 96 CTAs 68 us, 152 CTAs 102 us).  Otherwise one CTA per SM.
    const int sms = sm_count > 0 ? sm_count : kDefaultSmCount;
    long long g = sms;
    if (pl.n_tiles >= sms) {
      for (int c = sms; 2 * c >= sms; --c) {
        if (pl.n_tiles % c == 0) {
          g = c;
          break;
        }
      }
    }
    pl.blocks = (int)(g < pl.units ? g : pl.units);
  } else {
    if (blocks > pl.units) return W8A8_ERR_INVALID_ARG;
    pl.blocks = blocks;
  }
  if (pl.mma_n == 64) {
    pl.threads = tc::TcLayout<4>::kThreads;
    pl.stages = tc::TcLayout<4>::kWStages;
    pl.smem_bytes = tc::TcLayout<4>::kBytes;
  } else {
    pl.threads = tc::TcLayout<8>::kThreads;
    pl.stages = tc::TcLayout<8>::kWStages;
    pl.smem_bytes = tc::TcLayout<8>::kBytes;
  }
  pl.stage_units = tc::kStageUnits;
  // Workspace: header, counters, int32 planes, then the fp16 activations.  The counters and planes
  // are zero between calls and the activations are not, so every region sits at an offset that
  // does not depend on M: the planes are sized for MMA N = 128 whatever this call's M, and the
  // activations come last.  No call of either arm then finds its zeroed region written by another
  // (the decode arm's words, at most 32 KiB per 128 rows of N, end before the planes do).
  pl.counters_offset = kWsHeaderBytes;
  pl.partials_offset = pl.counters_offset + ((size_t)pl.n_tiles * sizeof(uint32_t) + 255) / 256 * 256;
  pl.x16_offset = pl.partials_offset + (size_t)pl.n_tiles * kTcMaxM * tc::kTileRows * sizeof(int);
  pl.workspace_bytes = pl.x16_offset + ((size_t)M * K * 2 + 255) / 256 * 256;
  *plan = pl;
  return W8A8_OK;
}

cudaError_t tc_launch(const TcPlan& pl, const int8_t* x, const float* xs, const void* wp, const float* wsc, void* out,
                      int M, int K, int N, void* ws, bool pdl, cudaStream_t stream, int* acc, bool stall) {
  uint8_t* const w = static_cast<uint8_t*>(ws);
  void* const x16 = w + pl.x16_offset;
  tc::TcParams p;
  // fp16 activations in the workspace (k permuted inside each 32-k unit, as the weight in tensor
  // memory): [M rows, K], box of 64 x mma_n (rows >= M read as 0).
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)tc::kBoxK, (cuuint32_t)pl.mma_n};
  const cuuint32_t estr[2] = {1u, 1u};
  cudaError_t e = encode_tensor_map_2d(&p.xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, dims, strides, box, estr,
                                       CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  p.wp = static_cast<const uint8_t*>(wp);
  p.x_scale = xs;
  p.w_scale = wsc;
  p.out = static_cast<uint16_t*>(out);
  p.status = reinterpret_cast<uint32_t*>(w);
  p.counters = reinterpret_cast<uint32_t*>(w + pl.counters_offset);
  p.planes = reinterpret_cast<int*>(w + pl.partials_offset);
  p.split = make_gemm_split(pl.n_tiles, pl.kb, pl.blocks);
  p.M = M;
  p.N = N;
  p.KB = pl.kb;
  p.tiles64 = pl.tiles64;
  p.acc_out = acc;
  p.debug_stall = stall ? 1 : 0;
  e = tc::launch_x16(x, x16, (long long)M * K / 32, pdl, stream);
  if (e != cudaSuccess) return e;
  return pl.mma_n == 64 ? tc::launch_tc<4>(p, pl.blocks, stream) : tc::launch_tc<8>(p, pl.blocks, stream);
}

}  // namespace w8a8
