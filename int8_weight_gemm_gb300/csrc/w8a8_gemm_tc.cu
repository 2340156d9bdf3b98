// W8A8 GEMM for 32 < M <= 128 on the fifth-generation tensor cores (tcgen05, sm_103a):
// out[M,N] = bf16((float(x_q @ W) * x_scale) * w_scale), the same operator and the same packed
// weight as the decode kernel.
//
// Operator: "INT8 W8A8 GEMM - Decode (M <= 32) - gfx928 / SGLang TP4", header paragraph.  Its
// section 3 ("Boundary: 16 < M <= 32") keeps a staged arm for larger M next to the decode arm, for
// the same (K, N): the decode pattern does not carry over once M grows.  This file is that arm.
// Split-K and the last-arrival combine follow the page's section 1.1 (qkv recipe): monotonic
// work split over the SM count, per-tile arrival counters in the workspace, the last arriver sums
// the partials, scales them and stores bf16, and every call leaves the workspace zeroed.
//
// Why tcgen05 here.  With M activation rows, every weight byte feeds 2M multiply-adds; at M = 128
// a weight stream at HBM speed needs ~1.8 PFLOP/s, three times what the register-fed mma.sync path
// of this part sustains, so the multiply moves to tcgen05.mma (M = 128 weight rows, N = 64 or 128
// activation rows, K = 16, f32 accumulation in tensor memory).  int8 tensor MMAs do not exist on
// sm_103a (ptxas rejects kind::i8), so every int8 is converted exactly to fp16 (each int8 value
// is an fp16 integer) and multiplied with kind::f16.
//
// Exactness.  A product is an integer of magnitude <= 2^14; one accumulator collects at most
// 512 k (four stages) before the epilogue warps read it out, so every f32 accumulator value is an
// integer of magnitude <= 2^23 and exact.  The read-out converts it to int32 (exact) and adds it
// to int32 sums; split tiles add int32 partials.  The result is the int32 sum an int8 MMA would
// give, bit for bit, whatever the split.
//
// Roles (one CTA per SM, all of its tensor memory):
//  * producer (one thread): per stage of 128 k, two 1-D bulk copies of packed weight (the CTA's
//    128-row tile is two consecutive 64-row packed tiles) and one 2-D tensor-map box of
//    activations (128 bytes x N_mma rows, 128-byte swizzle, zero fill past M and K) into a ring;
//  * eight converter warps: the weight rows go into tensor memory as the fp16 A operand
//    (tcgen05.st, lane = row), the activations into shared memory as the fp16 B operand
//    (K-major, no swizzle).  The same warps retire each stage once its MMAs have completed (they
//    wait for that anyway before reusing its operand slot): at the end of a period they read the
//    accumulators out and keep int32 sums in registers (each warp one lane quarter and one half
//    of the columns), and at the end of a segment they store bf16 or add the split tile's
//    partial and, as the last arrival, finish it;
//  * one or two MMA-issuing threads (each takes every other k-step into its own accumulators).
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
constexpr int kHalfBytes = kStageUnits * kPackSlab;  // one packed tile's share of a stage: 8 KiB
constexpr int kWStage = 2 * kHalfBytes;              // 16 KiB of weight per stage
constexpr int kConvWarps = 8;                        // two per tensor-memory lane quarter
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kProducerWarp = kConvWarps;
constexpr int kMmaWarp = kProducerWarp + 1;          // first MMA-issuing warp; owns tensor memory
constexpr int kPeriodStages = 4;                     // stages per accumulator read-out (512 k)
constexpr int kTmemCols = 512;
constexpr int kACols = kStageK / 2;                  // tensor-memory columns of one A stage (fp16 pairs)
constexpr int kBSbo = (kStageK / 8) * 128;           // B operand: bytes between 8-row groups
constexpr int kConvBarrier = 1;                      // named barrier of the converter warps

template <int NT16>
struct TcLayout {
  static constexpr int kN = 16 * NT16;               // MMA N: activation rows (zero past M)
  // An MMA at N = 64 is short next to an issuing thread's per-instruction cost, so two threads
  // issue; at N = 128 one keeps the tensor core busy and the accumulators fill tensor memory.
  static constexpr int kIssuers = kN <= 64 ? 2 : 1;
  static constexpr int kRawStages = kN <= 64 ? 6 : 4;
  static constexpr int kOpStages = kN <= 64 ? 4 : 3;
  static constexpr int kXBox = kN * 128;              // raw activation box, 1 KiB multiple
  static constexpr int kRaw = kXBox + kWStage;        // one raw stage (box first: 1 KiB aligned)
  static constexpr int kBStage = kN * kStageK * 2;    // fp16 B operand of one stage
  static constexpr int kDCol0 = kOpStages * kACols;   // first accumulator column
  static constexpr int kThreads = 32 * (kMmaWarp + kIssuers);
  static constexpr int kBytes = 1024 + kRawStages * kRaw + kOpStages * kBStage;
  static constexpr int kXPieces = kN * (kStageK / 16) / (32 * kConvWarps);   // 16-byte pieces per thread
  static constexpr int kCols = kN / 2;                // accumulator columns per converter warp
  static_assert(kDCol0 + kIssuers * 2 * kN <= kTmemCols, "tensor-memory columns");
  static_assert(kBytes <= 232448 - 2048, "shared memory");
  static_assert(kXPieces * 32 * kConvWarps == kN * (kStageK / 16), "activation pieces");
};

struct TcParams {
  CUtensorMap xmap;     // x_q [M,K] int8, box 128 bytes x N_mma rows, 128-byte swizzle
  const uint8_t* wp;    // packed weight (64-row tiles of 2 KiB slabs)
  const float* x_scale;
  const float* w_scale;
  uint16_t* out;
  uint32_t* status;
  uint32_t* counters;   // [tile] arrivals at a split tile, zero between calls
  int* planes;          // [tile][m < N_mma][row < 128] int32 sums of a split tile, zero between calls
  GemmSplit split;      // over the 128-row tiles, in 32-k units
  int M, N, KB, tiles64;
  int pdl;
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

// mbar_wait taken by a whole warp: the warp goes on only if every lane saw the phase complete, so
// the warp-wide tensor-memory instructions after it always run with all 32 lanes.
__device__ __forceinline__ bool mbar_wait_all(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status) {
  const bool ok = mbar_wait(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Bounded wait of all converter threads on one phase of `bar` (count kConvThreads).
__device__ __forceinline__ bool epi_sync(uint64_t* bar, uint32_t& phase, volatile int* abort, uint32_t* status) {
  mbar_arrive(bar);
  const bool ok = mbar_wait_all(bar, phase, abort, status);
  phase ^= 1u;
  return ok;
}

template <int NT16>
__global__ void __launch_bounds__(TcLayout<NT16>::kThreads, 1) w8a8_gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using L = TcLayout<NT16>;
  constexpr int kN = L::kN;
  constexpr int kI = L::kIssuers;
  constexpr int NR = L::kRawStages;
  constexpr int NA = L::kOpStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NR];    // a raw stage landed (weight halves + activation box)
  __shared__ __align__(8) uint64_t empty_bar[NR];   // the converter warps have read a raw stage
  __shared__ __align__(8) uint64_t conv_bar[NA];    // A (tensor memory) and B (shared memory) written
  __shared__ __align__(8) uint64_t mma_bar[NA];     // the MMAs reading an operand stage completed
  __shared__ __align__(8) uint64_t dempty_bar[2];   // an accumulator buffer has been read out
  __shared__ __align__(8) uint64_t final_bar[kI];   // every MMA of an issuer completed
  __shared__ __align__(8) uint64_t sync_bar;        // converter warps meet at a split tile's combine
  __shared__ uint32_t tmem_base;
  __shared__ float xs_sm[kN];
  __shared__ int abort_flag;
  __shared__ uint32_t last_flag;

  uint8_t* const smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* const raw = smem;                        // NR x [activation box | weight half 0 | weight half 1]
  uint8_t* const bring = smem + NR * L::kRaw;       // NA x fp16 B operand

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NR; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConvWarps);
    }
#pragma unroll
    for (int a = 0; a < NA; ++a) {
      mbar_init(&conv_bar[a], kConvThreads);
      mbar_init(&mma_bar[a], kI);
    }
#pragma unroll
    for (int d = 0; d < 2; ++d) mbar_init(&dempty_bar[d], kConvThreads);
#pragma unroll
    for (int i = 0; i < kI; ++i) mbar_init(&final_bar[i], 1);
    mbar_init(&sync_bar, kConvThreads);
    abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();   // the next call on the stream may start its own weight prefetch
  const uint32_t tmem = tmem_base;

  int b0, b1;
  gemm_split_run(p.split, blockIdx.x, &b0, &b1);

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer (one thread)
    if (lane == 0) {
      tma_prefetch_desc(&p.xmap);
      const uint64_t policy = policy_evict_first();
      // Weight halves of stage `w` into raw slot s; the expected bytes include the activation box.
      auto issue_w = [&](int s, const Walk& w) {
        const int t64 = 2 * w.t;
        const bool two = t64 + 1 < p.tiles64;
        const uint32_t bytes = (uint32_t)(w.ns * kPackSlab);
        mbar_arrive_expect_tx(&full_bar[s], bytes * (two ? 2u : 1u) + (uint32_t)L::kXBox);
        uint8_t* dst = raw + s * L::kRaw + L::kXBox;
        const uint8_t* src = p.wp + ((size_t)t64 * p.KB + w.kb0()) * kPackSlab;
        bulk_g2s_hint(dst, src, bytes, &full_bar[s], policy);
        if (two) bulk_g2s_hint(dst + kHalfBytes, src + (size_t)p.KB * kPackSlab, bytes, &full_bar[s], policy);
      };
      auto issue_x = [&](int s, const Walk& w) {
        tma_load_2d(raw + s * L::kRaw, &p.xmap, w.kb0() * kKBlock, 0, &full_bar[s]);
      };
      Walk it(b0, b1, p.KB);
      int q = 0;
      if (p.pdl) {
        // The packed weight is never written by the work this call depends on: stream it before the
        // dependency wait, and add the activation boxes once the wait has returned.
        Walk pre = it;
        int npre = 0;
        for (; npre < NR && !pre.done(); ++npre, pre.next()) issue_w(npre, pre);
        pdl_wait();
        for (; q < npre; ++q, it.next()) issue_x(q, it);
      } else {
        pdl_wait();
      }
      for (; !it.done(); it.next(), ++q) {
        const int s = q % NR;
        if (q >= NR && !mbar_wait(&empty_bar[s], (uint32_t)(((q / NR) & 1) ^ 1), &abort_flag, p.status)) break;
        issue_w(s, it);
        issue_x(s, it);
      }
      // Every copy issued must land before the CTA may exit.
      for (int s = 0; s < NR && s < q; ++s) {
        const int last = s + NR * ((q - 1 - s) / NR);
        mbar_wait_drain(&full_bar[s], (uint32_t)((last / NR) & 1), p.status);
      }
    }
  } else if (warp >= kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuers (one thread each)
    const int issuer = warp - kMmaWarp;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kTileRows, kN);
      bool started = false;   // this issuer's accumulator of the current period holds a k-step
      for (Walk it(b0, b1, p.KB); !it.done(); it.next()) {
        const int a = it.q % NA;
        const int db = it.period & 1;
        if (it.period_first() && it.period >= 2 &&
            !mbar_wait(&dempty_bar[db], (uint32_t)(((it.period >> 1) - 1) & 1), &abort_flag, p.status))
          break;
        if (!mbar_wait(&conv_bar[a], (uint32_t)((it.q / NA) & 1), &abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_addr = tmem + (uint32_t)(L::kDCol0 + (issuer * 2 + db) * kN);
        const uint32_t a_addr = tmem + (uint32_t)(a * kACols);
        const uint32_t b_addr = smem_addr(bring + a * L::kBStage);
        if (it.period_first()) started = false;
        // k-step j covers k in [16 j, 16 j + 16) of the stage: A columns 8 j ... 8 j + 7, B core
        // matrices 2 j and 2 j + 1 (128 bytes apart), 8-row groups kBSbo bytes apart.  Every issuer
        // has at least one k-step per stage (a stage has 2 ns >= 2 of them).
        for (int j = issuer; j < 2 * it.ns; j += kI) {
          umma_f16_tmem_a(d_addr, a_addr + 8u * j, smem_desc_kmajor(b_addr + 256u * j, 128u, (uint32_t)kBSbo), idesc,
                          started);
          started = true;
        }
        // Completes once these MMAs (and every earlier one of this thread) have completed: frees the
        // operand stage and, at a period's end, lets the converter warps read the accumulators.
        umma_commit(&mma_bar[a]);
      }
      // Whatever happened above, every MMA this thread issued completes before tensor memory is freed.
      umma_commit(&final_bar[issuer]);
      mbar_wait_drain(&final_bar[issuer], 0, p.status);
    }
  } else {
    // ---------------------------------------------------------------- converter warps
    // Warp w owns tensor-memory lanes 32 (w % 4) ... + 31 (rows of the CTA tile), units
    // 2 (w / 4), 2 (w / 4) + 1 of every stage, and accumulator columns (w / 4) kN / 2 ... + kN / 2 - 1.
    // Row r of the tile is row r % 64 = 16 s + g + 8 j of packed tile r / 64; a packed 16-byte
    // chunk (s, 4 g + c) holds k = 8c ... 8c + 7 of rows g and g + 8 (words: row g k 8c.., row
    // g + 8 k 8c.., row g k 8c+4.., row g + 8 k 8c+4..).  The two threads of rows g and g + 8
    // (lanes L and L ^ 8) each read two of the four chunks of their pair, trade the other row's
    // words, convert their own row's 32 values and write them as 16 fp16 pairs (tcgen05.st, columns
    // in k order).  Chunk choice by bit 1 of g spreads a quarter warp's reads over four bank groups.
    // The 256 converter threads also turn the stage's raw activation box into the fp16 B operand:
    // element (m, k) at (m / 8) kBSbo + (k / 8) 128 + (m % 8) 16 + (k % 8) 2.
    const int quad = warp & 3, upair = warp >> 2;
    const int half = quad >> 1;
    const int s16 = 2 * (quad & 1) + (lane >> 4);
    const int g = lane & 7;
    const bool jr = ((lane >> 3) & 1) != 0;
    const bool bsw = ((g >> 1) & 1) != 0;
    const int cA = 2 * (int)jr + (int)bsw, cB = 2 * (int)jr + 1 - (int)bsw;
    const int offA = (s16 * 32 + 4 * g + cA) * 16, offB = (s16 * 32 + 4 * g + cB) * 16;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * quad) << 16);
    const int row = 32 * quad + lane;
    const int m0 = upair * L::kCols;

    pdl_wait();   // x_scale, w_scale, out and the workspace may belong to the previous call
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
        mbar_arrive(&dempty_bar[db]);
        if (dr.seg_last()) {
          // Element (m0 + c, n) of out, walked down the column one activation row at a time.
          uint16_t* o = p.out + (size_t)m0 * p.N + n;
          const int mrows = min(L::kCols, p.M - m0);   // rows of this thread's half that exist
          if (dr.whole_tile()) {
            if (n < p.N) {
#pragma unroll
              for (int c = 0; c < L::kCols; ++c, o += p.N)
                if (c < mrows) *o = epilogue(iacc[c], xs_sm[m0 + c], wsv);
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
            if (!epi_sync(&sync_bar, sync_phase, &abort_flag, p.status)) return false;
            if (threadIdx.x == 0) {
              const uint32_t arrivals = (uint32_t)gemm_split_contributors(p.split, dr.t);
              const uint32_t old = atom_add_acq_rel_u32(p.counters + dr.t, 1u);
              if (old >= arrivals) atomicOr(p.status, W8A8_DEV_COUNTER_CORRUPT);
              const uint32_t last = old == arrivals - 1 ? 1u : 0u;
              if (last) p.counters[dr.t] = 0u;   // every contributor has arrived: ready for the next call
              last_flag = last;
            }
            if (!epi_sync(&sync_bar, sync_phase, &abort_flag, p.status)) return false;
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
    for (Walk it(b0, b1, p.KB); ok && !it.done(); it.next()) {
      const int s = it.q % NR;
      const int a = it.q % NA;
      if (!mbar_wait_all(&full_bar[s], (uint32_t)((it.q / NR) & 1), &abort_flag, p.status)) {
        ok = false;
        break;
      }
      if (it.q >= NA) {
        // The operand slot is free once the MMAs of stage q - NA have completed; that stage retires now.
        if (!mbar_wait_all(&mma_bar[a], (uint32_t)(((it.q - NA) / NA) & 1), &abort_flag, p.status) || !retire()) {
          ok = false;
          break;
        }
      }
      const bool have = 2 * it.t + half < p.tiles64;   // this packed tile exists (warp-uniform)
      const uint8_t* wsrc = raw + s * L::kRaw + L::kXBox + half * kHalfBytes;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int unit = 2 * upair + jj;
        if (!(have && unit < it.ns)) continue;
        const uint4 u = lds128(wsrc + unit * kPackSlab + offA);
        const uint4 v = lds128(wsrc + unit * kPackSlab + offB);
        // own row's words of chunks cA and cB, and the partner row's
        const uint32_t oa_lo = jr ? u.y : u.x, oa_hi = jr ? u.w : u.z;
        const uint32_t ob_lo = jr ? v.y : v.x, ob_hi = jr ? v.w : v.z;
        const uint32_t pa_lo = jr ? u.x : u.y, pa_hi = jr ? u.z : u.w;
        const uint32_t pb_lo = jr ? v.x : v.y, pb_hi = jr ? v.z : v.w;
        // this row's words of the partner's chunks 2 (1 - j) + bsw and 2 (1 - j) + 1 - bsw
        const uint32_t ra_lo = __shfl_xor_sync(0xffffffffu, pa_lo, 8);
        const uint32_t ra_hi = __shfl_xor_sync(0xffffffffu, pa_hi, 8);
        const uint32_t rb_lo = __shfl_xor_sync(0xffffffffu, pb_lo, 8);
        const uint32_t rb_hi = __shfl_xor_sync(0xffffffffu, pb_hi, 8);
        // chunks 2 j, 2 j + 1 (own) and 2 (1 - j), 2 (1 - j) + 1 (received), each in k order
        const uint32_t e0l = bsw ? ob_lo : oa_lo, e0h = bsw ? ob_hi : oa_hi;
        const uint32_t e1l = bsw ? oa_lo : ob_lo, e1h = bsw ? oa_hi : ob_hi;
        const uint32_t f0l = bsw ? rb_lo : ra_lo, f0h = bsw ? rb_hi : ra_hi;
        const uint32_t f1l = bsw ? ra_lo : rb_lo, f1h = bsw ? ra_hi : rb_hi;
        const uint32_t w[8] = {jr ? f0l : e0l, jr ? f0h : e0h, jr ? f1l : e1l, jr ? f1h : e1h,
                               jr ? e0l : f0l, jr ? e0h : f0h, jr ? e1l : f1l, jr ? e1h : f1h};
        uint32_t h[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) offset_bytes_to_half2_pairs(w[i], h[2 * i], h[2 * i + 1]);
        tmem_st16(t_lane + (uint32_t)(a * kACols + 16 * unit), h);
      }
      uint8_t* const bst = bring + a * L::kBStage;
#pragma unroll 2
      for (int rep = 0; rep < L::kXPieces; ++rep) {
        const int idx = threadIdx.x + kConvThreads * rep;
        const int m = idx % kN, pc = idx / kN;
        const uint4 xr = lds128(raw + s * L::kRaw + m * 128 + ((pc ^ (m & 7)) << 4));
        uint4 h0, h1;
        offset_bytes_to_half2_pairs(xr.x ^ 0x80808080u, h0.x, h0.y);
        offset_bytes_to_half2_pairs(xr.y ^ 0x80808080u, h0.z, h0.w);
        offset_bytes_to_half2_pairs(xr.z ^ 0x80808080u, h1.x, h1.y);
        offset_bytes_to_half2_pairs(xr.w ^ 0x80808080u, h1.z, h1.w);
        uint8_t* dst = bst + (m >> 3) * kBSbo + (2 * pc) * 128 + (m & 7) * 16;
        *reinterpret_cast<uint4*>(dst) = h0;
        *reinterpret_cast<uint4*>(dst + 128) = h1;
      }
      // Every raw value of the stage has been read and used.
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
      tmem_wait_st();
      fence_async_shared();
      tc_fence_before();
      mbar_arrive(&conv_bar[a]);
    }
    // Retire the stages still in flight.
    while (ok && !dr.done()) {
      if (!mbar_wait_all(&mma_bar[dr.q % NA], (uint32_t)((dr.q / NA) & 1), &abort_flag, p.status) || !retire()) break;
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
static cudaError_t launch_tc(const TcParams& p, int blocks, bool pdl, cudaStream_t stream) {
  auto kern = w8a8_gemm_tc_kernel<NT16>;
  const int smem = TcLayout<NT16>::kBytes;
  cudaError_t e = ensure_smem_attribute((const void*)kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(TcLayout<NT16>::kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, p);
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
    // One CTA per SM: each holds all of its SM's tensor memory and most of its shared memory.
    const long long g = sm_count > 0 ? sm_count : 152;
    pl.blocks = (int)(g < pl.units ? g : pl.units);
  } else {
    if (blocks > pl.units) return W8A8_ERR_INVALID_ARG;
    pl.blocks = blocks;
  }
  if (pl.mma_n == 64) {
    pl.threads = tc::TcLayout<4>::kThreads;
    pl.stages = tc::TcLayout<4>::kRawStages;
    pl.smem_bytes = tc::TcLayout<4>::kBytes;
  } else {
    pl.threads = tc::TcLayout<8>::kThreads;
    pl.stages = tc::TcLayout<8>::kRawStages;
    pl.smem_bytes = tc::TcLayout<8>::kBytes;
  }
  pl.stage_units = tc::kStageUnits;
  pl.counters_offset = kWsHeaderBytes;
  pl.partials_offset = pl.counters_offset + ((size_t)pl.n_tiles * sizeof(uint32_t) + 255) / 256 * 256;
  pl.workspace_bytes = pl.partials_offset + (size_t)pl.n_tiles * pl.mma_n * tc::kTileRows * sizeof(int);
  *plan = pl;
  return W8A8_OK;
}

cudaError_t tc_launch(const TcPlan& pl, const int8_t* x, const float* xs, const void* wp, const float* wsc, void* out,
                      int M, int K, int N, void* ws, bool pdl, cudaStream_t stream) {
  tc::TcParams p;
  // Activation tensor map: [M rows, K bytes], box of 128 bytes x mma_n rows (rows >= M read as 0).
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {128u, (cuuint32_t)pl.mma_n};
  const cuuint32_t estr[2] = {1u, 1u};
  cudaError_t e = encode_tensor_map_2d(&p.xmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<int8_t*>(x), dims, strides,
                                       box, estr, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  uint8_t* const w = static_cast<uint8_t*>(ws);
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
  p.pdl = pdl ? 1 : 0;
  return pl.mma_n == 64 ? tc::launch_tc<4>(p, pl.blocks, pdl, stream) : tc::launch_tc<8>(p, pl.blocks, pdl, stream);
}

}  // namespace w8a8
