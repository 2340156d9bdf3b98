// W8A8 decode GEMM for sm_103a: out[M,N] = bf16((float(x_q @ W) * x_scale) * w_scale), M <= 32.
//
// Operator: "INT8 W8A8 GEMM - Decode (M <= 32) - gfx928 / SGLang TP4", header paragraph.
// Structure follows that page's section 1.1 recipes and cross-shape rules, re-planned for GB300:
//  * the weight is packed once into the fragment layout (third cross-shape rule) so that the
//    kernel streams it as one contiguous byte range per CTA;
//  * split-K over a CTA count tied to the SM count (first rule), generalised to equal runs of
//    2 KiB slabs over the linearised (tile, k-block) space, all cuts on 32-aligned k;
//  * a fused last-arrival combine in one launch (qkv recipe: the last arriver at a split tile
//    holds the complete sum, scales it and stores bf16).  The recipe's per-tile counter, fence
//    and read-back become one returning 64-bit atomic per output element that carries both the
//    arrival count and the biased int32 sum, spread over all consumer threads;
//  * exact int32 sums, k-ascending within a split and ascending over splits.
//
// GB300 choices (prior art on the pages is gfx928 DUMMA; none of it carries over literally):
//  * The weight stream goes HBM -> shared memory through the TMA engine (cp.async.bulk, 1-D,
//    evict-first L2 policy) into an NS-deep ring of stages, issued by one producer warp.
//  * int8 tensor-core throughput on this part is far below what a weight stream at HBM speed
//    needs at M = 16 (measured with w8a8_mma_rate_probe: mma.sync s8 158 TOPS against fp16
//    587 TFLOPS), so the products run on the fp16 tensor path with fp32 accumulation: each
//    activation int8 becomes the fp16 integer it is, and each weight byte, stored offset binary
//    (w + 128), becomes the fp16 subnormal (w + 128) * 2^-24 with one byte permute (see
//    offset_bytes_to_subnormal_pairs).  Every fp32 partial over a window of at most 512 k is then
//    an exact multiple of 2^-24 below 1; windows are converted to int32 exactly and summed in
//    int32, and 128 * sum_k x comes off once per tile segment.  The result is the int32 sum an
//    int8 MMA would produce, bit for bit.
//  * Weight rows are the MMA's M dimension (16 rows per warp) and the activation rows are its
//    N dimension (n8 tiles), so M <= 8 wastes nothing on a 16-row MMA tile.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace w8a8 {

constexpr int kTileRows = 64;                      // rows of N per tile
constexpr int kKBlock = 32;                        // k per slab
constexpr int kSlabBytes = kTileRows * kKBlock;    // 2048
constexpr int kConsumerWarps = 8;                  // two per stage slot: even / odd stages
constexpr int kWarpsPerStage = 4;                  // one slab of a stage each
constexpr int kSubTiles = 4;                       // 16-row sub-tiles of a 64-row tile
constexpr int kThreads = 32 * (kConsumerWarps + 2);   // + one producer warp + one combine warp
// A launch whose CTAs each finish a single tile segment (the tile-aligned split) has nothing for
// the combine warp to do and leaves it out.
constexpr int kThreadsNoCombine = 32 * (kConsumerWarps + 1);
// 16 slabs of 32 k = 512 k per warp between int32 flushes: a window's fp32 partial stays an exact
// integer multiple of 2^-24 below 1 in magnitude (see offset_bytes_to_subnormal_pairs).
constexpr int kFlushSlabs = 16;

constexpr int kStageSlabs = 4;                     // one slab per consumer warp per stage

template <int NT8, int NS>
struct GemmLayout {
  static_assert(kStageSlabs * kKBlock == 128, "the activation box row is one 128-byte swizzle span");
  // Consumer warps split the stages by parity.  With an even ring depth every ring slot always holds
  // stages of one parity, so each warp waits on every phase of its slots' barriers; with an odd
  // depth a warp would skip phases and could not tell phase n from phase n + 2.
  static_assert(NS % 2 == 0, "the ring depth must be even");
  static constexpr int kXRows = 8 * NT8;                    // activation rows loaded (zero past M)
  static constexpr int kXRawStage = kXRows * 128;           // raw int8 box, 128B-swizzled, 1 KiB multiple
  static constexpr int kWStage = kStageSlabs * kSlabBytes;
  static constexpr int kSegSumInts = 2 * 4 * NT8 * 4 * 32;  // two int32 [sub][j][r][lane] segment sums
  static constexpr int kBytes = 1024 + NS * (kXRawStage + kWStage) + kSegSumInts * 4;   // + alignment slack
};

// --------------------------------------------------------------------------------------------
// Pack: W[K,N] row-major int8 -> packed slabs (layout documented in w8a8.h).
// --------------------------------------------------------------------------------------------
__global__ void w8a8_pack_kernel(const int8_t* __restrict__ W, int K, int N, int KB, long long chunks,
                                 uint4* __restrict__ out) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < chunks; idx += stride) {
    const int lane = (int)(idx & 31);
    long long r = idx >> 5;
    const int s = (int)(r & 3);
    r >>= 2;
    const int kb = (int)(r % KB);
    const long long t = r / KB;
    const int g = lane >> 2, c = lane & 3;
    uint32_t words[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const long long n = 64 * t + 16 * s + g + 8 * (w & 1);
      const int kbase = 32 * kb + 8 * c + 4 * (w >> 1);
      uint32_t v = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = n < N ? (uint32_t)(uint8_t)W[(long long)(kbase + b) * N + n] ^ 0x80u : 0x80u;
        v |= byte << (8 * b);
      }
      words[w] = v;
    }
    out[idx] = make_uint4(words[0], words[1], words[2], words[3]);
  }
}

// --------------------------------------------------------------------------------------------
// GEMM
// --------------------------------------------------------------------------------------------
struct GemmParams {
  // What a CTA needs before its first copy comes first, in one 64-byte line of the parameter
  // bank: each first touch of a line costs a constant-cache miss at launch.
  const uint8_t* wp;
  GemmSplit split;    // which slabs each CTA streams
  int KB;
  int pdl;            // W8A8_FLAG_PDL: the weight stream may start before the dependency wait
  int M, N;
  CUtensorMap xmap;   // x_q [M, K] int8, box 128 x (8 * NT8), 128-byte swizzle, zero fill past M
  const float* x_scale;
  const float* w_scale;
  uint16_t* out;
  uint32_t* status;
  // Split-tile combine words, zero between calls, layout [tile][sub-tile][n8 tile][fragment
  // register][lane].  pack_f = 0: one element per word, (arrivals << 52) + the sum of
  // (partial + 2^31).  pack_f = f > 0: elements e and e + half share the word of e, holding
  // a + b * 2^f + arrivals * 2^(2f) in two's complement, which every partial sum of the tile keeps
  // in range (see gemm_plan).
  unsigned long long* tile_acc;
  int K;
  int pack_f;
  int* acc_out;       // optional: the exact int32 sums [M, N] row-major, stored beside out
  int debug_stall;    // test hook: one warp of CTA 0 waits on a barrier that nothing completes
};

// A CTA's run of slabs [b0, b1) is cut by the tile boundaries into segments (one tile's part
// each).  Every segment but the last is finished by the combine warp (a round trip of returning
// atomics for a split tile) while the consumer warps stream on, so the segment walked last should
// be long enough to cover that work.  With tiles of at least 128 k-blocks (K >= 4096) the walk
// puts the longer of two segments last, and walks three as first, last, then the whole tile in
// the middle: measured on GB300 0.5 us less per call than the natural order at K = 4096,
// N = 24576, M = 16 (1.2 us together with the 4-slab run unit of make_gemm_split, 2.7 us at
// M = 32), and less at K = 8192 as well.  Shorter tiles keep the natural order: moving a whole
// tile last there made the second sum buffer wait for the first segment's combine behind a short
// segment (0.5-0.9 us slower at K = 2048 and K = 1024).
// Slab indices fit in 32 bits (at most 2^14 tiles x 2^11 k-blocks).
// multi = false: the launch's split gives every CTA a single segment (the tile-aligned split), a
// compile-time fact that leaves nothing to order.
struct RunOrder {
  int b0, b1, KB, t0, nseg, last;   // last: the segment (natural index) walked last
  __device__ RunOrder(int b0_, int b1_, int KB_, bool multi) : b0(b0_), b1(b1_), KB(KB_) {
    t0 = b0 / KB;
    if (!multi) {
      nseg = 1;
      last = 0;
      return;
    }
    nseg = b1 > b0 ? (b1 - 1) / KB - t0 + 1 : 0;
    last = nseg - 1;
    if (KB >= 128 && nseg == 2 && (t0 + 1) * KB - b0 > b1 - (t0 + 1) * KB) last = 0;
    if (KB >= 128 && nseg == 3) last = 1;
  }
  // Segment (in natural order) walked k-th.
  __device__ int index(int k) const { return k == nseg - 1 ? last : (k < last ? k : k + 1); }
  __device__ int begin(int i) const { return max(b0, (t0 + i) * KB); }
  __device__ int end(int i) const { return min(b1, (t0 + i + 1) * KB); }
};

// Walks the run as stages of at most SS slabs that never cross a tile, segment by segment in the
// order of RunOrder.
struct StageIter {
  RunOrder ro;
  int k, u, seg_end, t, ns, ss;
  __device__ StageIter(int b0_, int b1_, int KB_, int ss_, bool multi) : ro(b0_, b1_, KB_, multi), k(0), ss(ss_) {
    if (ro.nseg > 0) begin_segment();
  }
  __device__ void begin_segment() {
    const int i = ro.index(k);
    t = ro.t0 + i;
    u = ro.begin(i);
    seg_end = ro.end(i);
    ns = min(ss, seg_end - u);
  }
  __device__ bool done() const { return k >= ro.nseg; }
  __device__ int kb0() const { return u - t * ro.KB; }
  __device__ void next() {
    u += ns;
    if (u < seg_end) {
      ns = min(ss, seg_end - u);
    } else if (++k < ro.nseg) {
      begin_segment();
    }
  }
};

// Index of a fragment value in a segment sum (shared) or a tile accumulator (global): lanes are
// innermost, so a warp's 32 accesses of one (sub-tile, n8 tile, register) are contiguous.
template <int NT8>
__device__ __forceinline__ int frag_index(int u, int j, int r, int lane) {
  return ((u * NT8 + j) * 4 + r) * 32 + lane;
}

// Weight operand.  The packed bytes are offset binary, b = w + 128 in [0, 255].  With a zero high
// byte, the 16-bit pattern b is the fp16 subnormal b * 2^-24 (exponent field 0, significand b), so
// one byte permute builds two MMA operands and nothing is subtracted: the MMA then sums
// (w + 128) * x * 2^-24, and the 128 * sum_k x[m][k] it adds is taken off once per tile segment
// from the activation sums (segment_total).  lo receives bytes (0, 2), hi bytes (1, 3), each as
// (low half, high half).  Exactness: |(w + 128) x| <= 255 * 128 < 2^15, so a partial over at most
// 512 k is a multiple of 2^-24 below 1 in magnitude; fp32 holds every such value exactly, and the
// tensor pipe keeps fp16 subnormal operands (checked bit for bit on GB300 over 512-k windows at
// both ends of the range).
__device__ __forceinline__ void offset_bytes_to_subnormal_pairs(uint32_t u, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(u, 0u, 0x4240);
  hi = __byte_perm(u, 0u, 0x4341);
}

// A window's fp32 partial (an integer multiple of 2^-24, below 1 in magnitude) as the int32
// count of 2^-24 units: the scaling by 2^24 is exact and so is the conversion of an integral value.
__device__ __forceinline__ int window_to_int(float v) { return __float2int_rn(__fmul_rn(v, 16777216.0f)); }

// Split-tile combine words (see GemmParams::tile_acc).  Two-element word of f-bit fields: the
// increment of one CTA's partials (a, b), and the decode of a word into the sums a, b of the
// partials it holds and their count (a = the low f bits sign-extended, b = the next f bits
// sign-extended after removing a, the count = the rest after removing b).
__device__ __forceinline__ unsigned long long pair_increment(int va, int vb, int f) {
  return (1ull << (2 * f)) + ((unsigned long long)(long long)vb << f) + (unsigned long long)(long long)va;
}
__device__ __forceinline__ uint32_t pair_decode(unsigned long long w, int f, long long* a, long long* b) {
  const unsigned long long mask = (1ull << f) - 1ull;
  const int sh = 64 - f;
  *a = (long long)((w & mask) << sh) >> sh;
  const unsigned long long w1 = (w - (unsigned long long)*a) >> f;
  *b = (long long)((w1 & mask) << sh) >> sh;
  return (uint32_t)((w1 - (unsigned long long)*b) >> f);
}
// One-element word: (arrivals << 52) + the sum of (partial + 2^31); the total of n partials is the
// low 32 bits minus n * 2^31 (mod 2^32).
__device__ __forceinline__ unsigned long long single_increment(int v) {
  return (1ull << 52) + ((uint32_t)v ^ 0x80000000u);
}
__device__ __forceinline__ int single_total(unsigned long long old, int v, uint32_t n) {
  return (int)((uint32_t)old + ((uint32_t)v ^ 0x80000000u) - ((n & 1u) << 31));
}

// Epilogue of one output element: out[m][n] = bf16_rne((float(acc) * x_scale[m]) * w_scale[n]),
// and the int32 sum itself when the caller asked for it.
__device__ __forceinline__ void store_out(const GemmParams& p, int m, int n, int acc, float xsv, float wsv) {
  if (m < p.M && n < p.N) {
    float f = __int2float_rn(acc);
    f = __fmul_rn(f, xsv);
    f = __fmul_rn(f, wsv);
    p.out[(long long)m * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(f));
    if (p.acc_out) p.acc_out[(long long)m * p.N + n] = acc;
  }
}

constexpr int kProducerWarp = kConsumerWarps;        // warp 8: lane 0 issues every copy
constexpr int kProducerThread = 32 * kProducerWarp;
constexpr int kCombineWarp = kConsumerWarps + 1;     // warp 9: finishes every segment but a CTA's last
// Returning atomics the combine warp keeps in flight per lane (16 measured no faster).
constexpr int kCombineBatch = 8;
constexpr int kConsumerThreads = 32 * kConsumerWarps;

template <int NT8, int NS, bool kMulti>
// kMulti: some CTA finishes more than one tile segment (the run split), so a combine warp finishes
// every segment but a CTA's last; without it every CTA has exactly one segment.
__global__ void __launch_bounds__(kMulti ? kThreads : kThreadsNoCombine, 2)
    w8a8_gemm_kernel(const __grid_constant__ GemmParams p) {
  using L = GemmLayout<NT8, NS>;
  constexpr int kSegInts = L::kSegSumInts / 2;      // one segment-sum buffer
  constexpr int kPer = kSegInts / kConsumerThreads; // output elements per consumer thread at a segment end
  static_assert(kPer * kConsumerThreads == kSegInts, "segment sums split evenly over the consumers");
  // Work split of the consumer warps.  NT8 <= 2: warp w takes slab w % 4 of the stages of parity
  // w / 4, all four sub-tiles.  NT8 >= 3 (the accumulators of four sub-tiles would not fit the
  // register budget): warp w takes slab w % 4 of every stage, sub-tiles 2 (w / 4) and 2 (w / 4) + 1.
  constexpr bool kHalfSubTiles = NT8 >= 3;
  constexpr int kWarpSubTiles = kHalfSubTiles ? kSubTiles / 2 : kSubTiles;
  constexpr int kStageWarps = kHalfSubTiles ? kConsumerWarps : kWarpsPerStage;   // consumers of a stage
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NS];   // W slabs + raw activation box of a stage landed
  __shared__ __align__(8) uint64_t empty_bar[NS];  // the stage's consumer warps took their slabs
  __shared__ float xs_sm[32];                      // x_scale (0 past M)
  __shared__ float ws_sm[2][kTileRows];            // w_scale of a segment's tile, by segment parity
  __shared__ int xsum_sm[2][32];                   // sum_k x[m][k] over a segment's k, by segment parity
  __shared__ __align__(8) uint64_t seg_bar;        // every consumer warp finished the CTA's last segment
  __shared__ __align__(8) uint64_t seg_full[2];    // every consumer warp flushed an earlier segment (by parity)
  __shared__ __align__(8) uint64_t seg_free[2];    // the combine warp is done with that segment's buffer
  __shared__ __align__(8) uint64_t stall_bar;      // test hook only: never completed
  __shared__ int abort_flag;

  // 128B-swizzled TMA boxes need a 1 KiB aligned destination.
  uint8_t* const smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* const xraw = smem;
  uint8_t* const wring = xraw + NS * L::kXRawStage;
  int* const segsum = reinterpret_cast<int*>(wring + NS * L::kWStage);   // [2][sub][j][r][lane] int32

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int b0, b1;
  gemm_split_run(p.split, (int)blockIdx.x, &b0, &b1);

  // Every launch is a programmatic dependent of the work before it on the stream (gemm_launch), so
  // a CTA may start while the previous kernel finishes.  Until the dependency wait (griddepcontrol
  // .wait, after which that kernel's writes are visible) a CTA only sets itself up (parameters,
  // barriers, shared memory) and prefetches its first stages' weight bytes into L2.  With
  // W8A8_FLAG_PDL (p.pdl) the producer instead issues those stages' weight copies into shared
  // memory before the CTA-wide barrier, the caller having promised that nothing in flight writes
  // the weights; the activation boxes always wait.  Every copy of a stage lands on the
  // stage's full barrier, which counts the weight and activation bytes together.
  const uint32_t xbox = (uint32_t)L::kXRawStage;
  StageIter it(b0, b1, p.KB, kStageSlabs, kMulti);   // producer: the next stage to issue
  int pq = 0;                                 // producer: stages issued so far
  uint64_t policy = 0;
  if (threadIdx.x == kProducerThread) {
    tma_prefetch_desc(&p.xmap);
    policy = policy_evict_first();
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kStageWarps);
    }
    mbar_init(&seg_bar, kConsumerWarps);
    mbar_init(&seg_full[0], kConsumerWarps);
    mbar_init(&seg_full[1], kConsumerWarps);
    mbar_init(&seg_free[0], 1);
    mbar_init(&seg_free[1], 1);
    mbar_init(&stall_bar, 1);
    abort_flag = 0;
    mbar_fence_init();
    // The packed weight is never written by the work this call depends on, so its first stages
    // are requested at once; the activation boxes wait for the dependency when there is one.
    for (; p.pdl && pq < NS && !it.done(); it.next(), ++pq) {
      mbar_arrive_expect_tx(&full_bar[pq], (uint32_t)(it.ns * kSlabBytes) + xbox);
      bulk_g2s_hint(wring + pq * L::kWStage, p.wp + (size_t)it.u * kSlabBytes, (uint32_t)(it.ns * kSlabBytes),
                    &full_bar[pq], policy);
    }
    // Without that promise the first stages' weight bytes are only prefetched into L2, which
    // changes nothing a later read returns; the copies after the dependency wait then hit in L2.
    if (!p.pdl) {
      StageIter pf(b0, b1, p.KB, kStageSlabs, kMulti);
      for (int j = 0; j < NS && !pf.done(); pf.next(), ++j)
        bulk_prefetch_l2(p.wp + (size_t)pf.u * kSlabBytes, (uint32_t)(pf.ns * kSlabBytes));
    }
  }
  for (int i = threadIdx.x; i < L::kSegSumInts; i += (kMulti ? kThreads : kThreadsNoCombine)) segsum[i] = 0;
  if (threadIdx.x < 64) (&xsum_sm[0][0])[threadIdx.x] = 0;
  __syncthreads();
  pdl_trigger();   // the next call on the stream may start its own weight prefetch

  // Row m of element e of a segment's sums (layout [sub][j][r][lane]) and its column inside the
  // tile: the inverse of frag_index and of the accumulator fragment (lane = 4g + c holds rows
  // 2c + (r & 1) of n8 tile j and columns g + 8 (r >> 1) of sub-tile u).
  auto elem_m = [](int e) { return 8 * ((e >> 7) % NT8) + 2 * (e & 3) + ((e >> 5) & 1); };
  auto elem_n = [](int e) { return 16 * ((e >> 7) / NT8) + ((e & 31) >> 2) + 8 * ((e >> 6) & 1); };
  // The exact int32 sum of element e over this CTA's part of the segment in buffer b: the shared
  // sum holds sum (w + 128) x, and 128 * sum_k x[m][k] over the segment's k comes off here.
  auto segment_total = [&](int e, int b, int biased) { return biased - 128 * xsum_sm[b][elem_m(e)]; };
  // Store element e of tile t with its scales parked in buffer b.
  auto store_elem = [&](int e, int t, int b, int total) {
    const int m = elem_m(e), nl = elem_n(e);
    store_out(p, m, t * kTileRows + nl, total, xs_sm[m], ws_sm[b][nl]);
  };

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer (one thread)
    if (threadIdx.x != kProducerThread) return;
    pdl_wait();
    if (p.pdl) {
      // The activation boxes of the stages whose weight copies went out before the wait.
      StageIter pre(b0, b1, p.KB, kStageSlabs, kMulti);
      for (int j = 0; j < pq; pre.next(), ++j)
        tma_load_2d(xraw + j * L::kXRawStage, &p.xmap, pre.kb0() * kKBlock, 0, &full_bar[j]);
    } else {
      // The first ring of stages, weight and activations together, now that the previous kernel's
      // writes are visible.
      for (; pq < NS && !it.done(); it.next(), ++pq) {
        mbar_arrive_expect_tx(&full_bar[pq], (uint32_t)(it.ns * kSlabBytes) + xbox);
        bulk_g2s_hint(wring + pq * L::kWStage, p.wp + (size_t)it.u * kSlabBytes, (uint32_t)(it.ns * kSlabBytes),
                      &full_bar[pq], policy);
        tma_load_2d(xraw + pq * L::kXRawStage, &p.xmap, it.kb0() * kKBlock, 0, &full_bar[pq]);
      }
    }
    int s = pq % NS;                       // ring slot of stage pq
    uint32_t ph = (uint32_t)((pq / NS) & 1);   // its phase parity
    for (; !it.done(); it.next(), ++pq) {
      if (!mbar_wait(&empty_bar[s], ph ^ 1u, &abort_flag, p.status)) break;
      mbar_arrive_expect_tx(&full_bar[s], (uint32_t)(it.ns * kSlabBytes) + xbox);
      bulk_g2s_hint(wring + s * L::kWStage, p.wp + (size_t)it.u * kSlabBytes, (uint32_t)(it.ns * kSlabBytes), &full_bar[s],
                    policy);
      tma_load_2d(xraw + s * L::kXRawStage, &p.xmap, it.kb0() * kKBlock, 0, &full_bar[s]);
      if (++s == NS) {
        s = 0;
        ph ^= 1u;
      }
    }
    // Drain: every copy this thread issued must land before the CTA may exit.
    for (int d = 0; d < NS && d < pq; ++d) {
      const int last = d + NS * ((pq - 1 - d) / NS);
      mbar_wait_drain(&full_bar[d], (uint32_t)((last / NS) & 1), p.status);
    }
    return;
  }

  if (kMulti && warp == kCombineWarp) {
    // ---------------------------------------------------------------- combine warp
    // Finishes every segment of this CTA except its last: waits until the consumer warps have
    // flushed the segment's sums, stores a whole tile directly or adds a split tile's partials
    // into its workspace words (storing the elements this CTA completes), clears the sums and
    // hands the buffer back.  The consumer warps stream on meanwhile; the last segment, after
    // which there is nothing left to stream, they finish themselves.
    pdl_wait();   // out and the workspace words may belong to the previous call
    const RunOrder ro(b0, b1, p.KB, kMulti);
    for (int s = 0; s + 1 < ro.nseg; ++s) {
      const int si = ro.index(s);
      const int t = ro.t0 + si;
      const int seg_begin = ro.begin(si);
      const int buf = s & 1;
      if (!mbar_wait(&seg_full[buf], (uint32_t)((s >> 1) & 1), &abort_flag, p.status)) return;
      int* const sums = segsum + buf * kSegInts;
      unsigned long long* const tacc = p.tile_acc + (size_t)t * kSegInts;
      const uint32_t n = (uint32_t)gemm_split_contributors(p.split, t);
      if (seg_begin == t * p.KB && ro.end(si) == (t + 1) * p.KB) {   // the whole tile is ours
        for (int e = lane; e < kSegInts; e += 32) {
          store_elem(e, t, buf, segment_total(e, buf, sums[e]));
          sums[e] = 0;
        }
      } else if (p.pack_f) {
        constexpr int kHalf = kSegInts / 2, kWords = kHalf / 32;   // words of this lane: lane + 32 w
        for (int w0 = 0; w0 < kWords; w0 += kCombineBatch) {
          unsigned long long old[kCombineBatch];
#pragma unroll
          for (int k = 0; k < kCombineBatch; ++k) {
            const int i = lane + 32 * (w0 + k);
            if (w0 + k < kWords)
              old[k] = atom_add_relaxed_u64(tacc + i, pair_increment(segment_total(i, buf, sums[i]),
                                                                     segment_total(i + kHalf, buf, sums[i + kHalf]),
                                                                     p.pack_f));
          }
#pragma unroll
          for (int k = 0; k < kCombineBatch; ++k) {
            const int i = lane + 32 * (w0 + k);
            if (w0 + k >= kWords) break;
            long long a, bb;
            const uint32_t arrived = pair_decode(old[k], p.pack_f, &a, &bb);
            if (arrived == n - 1) {
              tacc[i] = 0ull;
              store_elem(i, t, buf, (int)(a + segment_total(i, buf, sums[i])));
              store_elem(i + kHalf, t, buf, (int)(bb + segment_total(i + kHalf, buf, sums[i + kHalf])));
            } else if (arrived >= n) {
              atomicOr(p.status, W8A8_DEV_COUNTER_CORRUPT);
            }
            sums[i] = 0;
            sums[i + kHalf] = 0;
          }
        }
      } else {
        constexpr int kElems = kSegInts / 32;
        for (int w0 = 0; w0 < kElems; w0 += kCombineBatch) {
          unsigned long long old[kCombineBatch];
#pragma unroll
          for (int k = 0; k < kCombineBatch; ++k) {
            const int e = lane + 32 * (w0 + k);
            if (w0 + k < kElems) old[k] = atom_add_relaxed_u64(tacc + e, single_increment(segment_total(e, buf, sums[e])));
          }
#pragma unroll
          for (int k = 0; k < kCombineBatch; ++k) {
            const int e = lane + 32 * (w0 + k);
            if (w0 + k >= kElems) break;
            const uint32_t arrived = (uint32_t)(old[k] >> 52);
            if (arrived == n - 1) {
              tacc[e] = 0ull;
              store_elem(e, t, buf, single_total(old[k], segment_total(e, buf, sums[e]), n));
            } else if (arrived >= n) {
              atomicOr(p.status, W8A8_DEV_COUNTER_CORRUPT);
            }
            sums[e] = 0;
          }
        }
      }
      __syncwarp();
      xsum_sm[buf][lane] = 0;   // every lane has read the activation sums of this buffer
      __syncwarp();
      if (lane == 0) mbar_arrive(&seg_free[buf]);
    }
    return;
  }

  // ---------------------------------------------------------------- consumer warps
  // Warp w multiplies slab (w % 4) of every stage of parity (w / 4), covering all four 16-row
  // sub-tiles of the 64-row tile.  Each warp converts only its own 32-k activation slice, so the
  // warps never wait for one another inside a tile.  Their fp32 partials (exact) are flushed as
  // int32 into the segment's shared sum buffer (two buffers, used by alternate segments), and the
  // lanes' activation sums go to the segment's xsum_sm.  At the end of each segment all consumer
  // threads finish it together: every thread takes kPer of its output elements (one returning
  // atomic each for a split tile), so the tail of a segment is one global round trip.  Meanwhile
  // the producer keeps filling the ring.
  pdl_wait();   // x_scale, w_scale, out and the accumulators may belong to the previous call
  if (p.debug_stall && blockIdx.x == 0 && warp == 0) {
    // Test hook of the device fault path: this warp waits, with a short bound, on a barrier that
    // nothing completes.  The wait runs out, records W8A8_DEV_WAIT_TIMEOUT and raises the abort
    // flag; the other roles of the CTA then give up at their next wait, the producer after
    // draining the copies it issued.  Nothing hangs and nothing faults.
    mbar_wait(&stall_bar, 0u, &abort_flag, p.status, kTestStallCycles);
    return;
  }
  const int g = lane >> 2, c = lane & 3;
  const int slab = warp & (kStageSlabs - 1);
  const int half = warp / kStageSlabs;
  const int sub0 = kHalfSubTiles ? kWarpSubTiles * half : 0;   // first sub-tile of this warp
  // The activation sums.  NT8 <= 2: each warp sums the rows of every n8 tile of its slabs.
  // NT8 >= 3: the two warps of a slab position see the same activations, so each sums half of
  // the n8 tiles (j in [xj0, xj0 + kXsumTiles)), which also halves the registers it needs.
  constexpr int kXsumTiles = kHalfSubTiles ? (NT8 + 1) / 2 : NT8;
  const int xj0 = kHalfSubTiles ? half * kXsumTiles : 0;
  float facc[kWarpSubTiles][NT8][4];
#pragma unroll
  for (int u = 0; u < kWarpSubTiles; ++u)
#pragma unroll
    for (int j = 0; j < NT8; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) facc[u][j][r] = 0.f;
  int xsum[kXsumTiles];   // sum of this lane's activation bytes of row 8 (xj0 + i) + g over the segment
#pragma unroll
  for (int i = 0; i < kXsumTiles; ++i) xsum[i] = 0;
  int since = 0;          // slabs accumulated in fp32 by this warp since its last flush
  int segs = 0;
  int q = 0;              // CTA-wide stage index of the current segment's first stage
  uint32_t arrivals = 0;  // CTAs whose runs share the current segment's tile
  // Scales are fetched into registers long before they are needed (x_scale at the start, a
  // tile's w_scale at the start of its segment) and parked in shared memory just before the
  // segment barrier: loads issued at the very end of the call, when every CTA issues them at
  // once, were measured to stall the epilogue for microseconds.
  const float xs_reg = threadIdx.x < 32 && (int)threadIdx.x < p.M ? __ldg(p.x_scale + threadIdx.x) : 0.f;
  float ws_reg = 0.f;
  // Add this warp's fp32 window partials (exact) into the segment's shared int32 sums.
  auto flush = [&](int* dst) {
#pragma unroll
    for (int u = 0; u < kWarpSubTiles; ++u)
#pragma unroll
      for (int j = 0; j < NT8; ++j)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          atomicAdd(dst + frag_index<NT8>(sub0 + u, j, r, lane), window_to_int(facc[u][j][r]));
          facc[u][j][r] = 0.f;
        }
  };

  // Output element i of this thread at the last segment's end: e = threadIdx.x + kConsumerThreads * i.
  auto finish = [&](int i, int t, int b, int total) { store_elem(threadIdx.x + kConsumerThreads * i, t, b, total); };

  // Offsets of this warp's fragments inside a stage (the same for every stage): W fragments of
  // its sub-tiles in its slab; row g of the activation box sits at g * 128 with its 16-byte chunks
  // XOR-swizzled by g, and n8 tile j adds j * 1024.
  const int w_off = slab * kSlabBytes + sub0 * 512 + lane * 16;
  const int x_off = g * 128 + (((2 * slab + (c >> 1)) ^ g) << 4) + 8 * (c & 1);
  constexpr int kStep = kHalfSubTiles ? 1 : 2;   // stages from one of this warp's stages to the next

  // The run [b0, b1) is walked segment by segment (one tile's part each, in RunOrder's order); a
  // segment of n slabs is ceil(n / 4) stages of the CTA-wide stage sequence, the last one possibly
  // partial.  q is the
  // CTA-wide index of the segment's first stage; this warp visits only its own stages nq, whose
  // ring slot and phase parity it keeps up to date as it goes.
  int nq = kHalfSubTiles ? 0 : half;   // next CTA-wide stage this warp visits (< NS here)
  int slot = nq;
  uint32_t phase = 0;
  const RunOrder ro(b0, b1, p.KB, kMulti);
  for (int k = 0; k < ro.nseg; ++k) {
    const int si = ro.index(k);
    const int t = ro.t0 + si;
    const int seg_begin = ro.begin(si), seg_end = ro.end(si);
    const int seg_slabs = seg_end - seg_begin;
    const int seg_stages = (seg_slabs + kStageSlabs - 1) / kStageSlabs;
    // Start of a segment: count the tile's contributors and fetch its w_scale now, off the
    // segment's tail.  The sum buffer of this segment's parity is free once the combine warp has
    // finished the segment two before (the last segment never shares its buffer with a later one).
    arrivals = (uint32_t)gemm_split_contributors(p.split, t);
    if (kMulti && segs >= 2 && !mbar_wait(&seg_free[segs & 1], (uint32_t)(((segs - 2) >> 1) & 1), &abort_flag, p.status))
      return;
    if (threadIdx.x < kTileRows) {
      const int n = t * kTileRows + (int)threadIdx.x;
      ws_reg = n < p.N ? __ldg(p.w_scale + n) : 0.f;
    }
    const int q_end = q + seg_stages;
    for (; nq < q_end; nq += kStep) {
      if (!mbar_wait(&full_bar[slot], phase, &abort_flag, p.status)) return;
      if (slab < seg_slabs - kStageSlabs * (nq - q)) {
        // Weight fragments of this warp's sub-tiles, then this slab's activation B fragments.
        const uint8_t* wst = wring + slot * L::kWStage + w_off;
        uint4 w[kWarpSubTiles];
#pragma unroll
        for (int u = 0; u < kWarpSubTiles; ++u) w[u] = *reinterpret_cast<const uint4*>(wst + u * 512);
        const uint8_t* xr = xraw + slot * L::kXRawStage + x_off;
        uint32_t b[NT8][4];
#pragma unroll
        for (int j = 0; j < NT8; ++j) {
          const uint2 v = *reinterpret_cast<const uint2*>(xr + j * 1024);
          offset_bytes_to_half2(v.x ^ 0x80808080u, b[j][0], b[j][1]);
          offset_bytes_to_half2(v.y ^ 0x80808080u, b[j][2], b[j][3]);
          if (!kHalfSubTiles) {
            xsum[j] = __dp4a((int)v.y, 0x01010101, __dp4a((int)v.x, 0x01010101, xsum[j]));
          } else {
#pragma unroll
            for (int i = 0; i < kXsumTiles; ++i)
              if (j == xj0 + i) xsum[i] = __dp4a((int)v.y, 0x01010101, __dp4a((int)v.x, 0x01010101, xsum[i]));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);   // registers hold everything this warp needs
        if (since == kFlushSlabs) {
          flush(segsum + (segs & 1) * kSegInts);
          since = 0;
        }
        // Sub-tile by sub-tile: its two k-steps' weight fragments, then its MMAs.  Only one
        // sub-tile's converted fragments are live at a time (measured fewer instructions and
        // 0.4 us less on the gate_up-sized call than converting all four first).
#pragma unroll
        for (int u = 0; u < kWarpSubTiles; ++u) {
          uint32_t a[2][4];
          offset_bytes_to_subnormal_pairs(w[u].x, a[0][0], a[0][2]);   // row g,   k 8c+0..3
          offset_bytes_to_subnormal_pairs(w[u].y, a[0][1], a[0][3]);   // row g+8, k 8c+0..3
          offset_bytes_to_subnormal_pairs(w[u].z, a[1][0], a[1][2]);   // row g,   k 8c+4..7
          offset_bytes_to_subnormal_pairs(w[u].w, a[1][1], a[1][3]);   // row g+8, k 8c+4..7
#pragma unroll
          for (int st = 0; st < 2; ++st)
#pragma unroll
            for (int j = 0; j < NT8; ++j)
              mma_f16_16816(facc[u][j], a[st][0], a[st][1], a[st][2], a[st][3], b[j][2 * st], b[j][2 * st + 1]);
        }
        ++since;
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
      }
      slot += kStep;
      if (slot >= NS) {
        slot -= NS;
        phase ^= 1u;
      }
    }
    q = q_end;

    // ------------------------------------------------------------ end of this CTA's part of a tile
    const int buf = segs & 1;
    if (threadIdx.x < 32 && segs == 0) xs_sm[threadIdx.x] = xs_reg;
    if (threadIdx.x < kTileRows) ws_sm[buf][threadIdx.x] = ws_reg;
    int* const sums = segsum + buf * kSegInts;
    if (since) flush(sums);
    since = 0;
    // Row 8j + g's activation sum over this warp's slabs: the four lanes of a row hold 32 k each.
#pragma unroll
    for (int i = 0; i < kXsumTiles; ++i) {
      int sx = xsum[i];
      sx += __shfl_xor_sync(0xffffffffu, sx, 1);
      sx += __shfl_xor_sync(0xffffffffu, sx, 2);
      if (c == 0 && xj0 + i < NT8) atomicAdd(&xsum_sm[buf][8 * (xj0 + i) + g], sx);
      xsum[i] = 0;
    }
    ++segs;
    if (kMulti && k + 1 < ro.nseg) {
      // An earlier segment: hand it to the combine warp and stream on.
      __syncwarp();
      if (lane == 0) mbar_arrive(&seg_full[buf]);
      continue;
    }
    // The last segment: every consumer's part is in the sums and the scales are in shared memory
    // once all consumer warps have met (an mbarrier wait, bounded like every other: a warp that
    // gave up on a timeout never arrives, and the others then give up too).  The consumers finish
    // it together, every thread kPer elements.
    __syncwarp();
    if (lane == 0) mbar_arrive(&seg_bar);
    if (!mbar_wait(&seg_bar, 0u, &abort_flag, p.status)) return;
    int* const mine = sums + threadIdx.x;   // element i at mine[kConsumerThreads * i]
    auto mine_total = [&](int i) { return segment_total(threadIdx.x + kConsumerThreads * i, buf, mine[kConsumerThreads * i]); };
    if (seg_begin == t * p.KB && seg_end == (t + 1) * p.KB) {   // the whole tile is ours
#pragma unroll
      for (int i = 0; i < kPer; ++i) finish(i, t, buf, mine_total(i));
      break;
    }
    // Split tile.  Each contributor adds its partials into the elements' workspace words with one
    // returning atomic per word; the contributor that brings a word's count to n holds the same
    // total, in the same bits, as an ascending-order sum of the n partials (int32 addition is
    // associative), stores the bf16 result and returns the word to zero for the next call.  No
    // separate counter, fence or read-back.  Two elements share a word when the fields fit
    // (pack_f), halving the atomics.
    unsigned long long* const tacc = p.tile_acc + (size_t)t * kSegInts + threadIdx.x;
    if (p.pack_f) {
      unsigned long long old[kPer / 2];
#pragma unroll
      for (int i = 0; i < kPer / 2; ++i)
        old[i] = atom_add_relaxed_u64(tacc + kConsumerThreads * i,
                                      pair_increment(mine_total(i), mine_total(i + kPer / 2), p.pack_f));
#pragma unroll
      for (int i = 0; i < kPer / 2; ++i) {
        long long a, bb;
        const uint32_t arrived = pair_decode(old[i], p.pack_f, &a, &bb);
        if (arrived == arrivals - 1) {
          tacc[kConsumerThreads * i] = 0ull;
          finish(i, t, buf, (int)(a + mine_total(i)));
          finish(i + kPer / 2, t, buf, (int)(bb + mine_total(i + kPer / 2)));
        } else if (arrived >= arrivals) {
          atomicOr(p.status, W8A8_DEV_COUNTER_CORRUPT);
        }
      }
    } else {
      unsigned long long old[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) old[i] = atom_add_relaxed_u64(tacc + kConsumerThreads * i, single_increment(mine_total(i)));
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const uint32_t arrived = (uint32_t)(old[i] >> 52);
        if (arrived == arrivals - 1) {
          tacc[kConsumerThreads * i] = 0ull;
          finish(i, t, buf, single_total(old[i], mine_total(i), arrivals));
        } else if (arrived >= arrivals) {
          atomicOr(p.status, W8A8_DEV_COUNTER_CORRUPT);
        }
      }
    }
  }
}

// --------------------------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------------------------
// Pipeline depth per n8-tile count, sized for two CTAs per SM.
constexpr int kStages1 = 10, kStages2 = 10, kStages3 = 8, kStages4 = 6;

static int gemm_stages(int nt8) {
  switch (nt8) {
    case 1: return kStages1;
    case 2: return kStages2;
    case 3: return kStages3;
    default: return kStages4;
  }
}

static size_t gemm_smem_bytes(int nt8) {
  switch (nt8) {
    case 1: return GemmLayout<1, kStages1>::kBytes;
    case 2: return GemmLayout<2, kStages2>::kBytes;
    case 3: return GemmLayout<3, kStages3>::kBytes;
    default: return GemmLayout<4, kStages4>::kBytes;
  }
}

static constexpr int kAutoCtasPerSm = 2;   // resident CTAs per SM (shared memory and registers)

int gemm_plan(int M, int K, int N, int blocks, int sm_count, GemmPlan* plan) {
  if (M < 1 || M > 32 || K < 1 || K > 65536 || N < 1 || N > 1048576 || blocks < 0) return W8A8_ERR_INVALID_ARG;
  if (K % 32 != 0 || N % 8 != 0) return W8A8_ERR_UNSUPPORTED_SHAPE;
  GemmPlan pl{};
  pl.nt8 = (M + 7) / 8;
  pl.n_tiles = (N + kTileRows - 1) / kTileRows;
  pl.kb = K / kKBlock;
  pl.slabs = (long long)pl.n_tiles * pl.kb;
  if (blocks == 0) {
    // Up to two CTAs on every SM (the most that fit): fewer CTAs than tiles stream slower and save
    // little in the split-tile combine, which costs one round trip.
    const long long g = (long long)kAutoCtasPerSm * (sm_count > 0 ? sm_count : 152);
    long long gg = g < pl.slabs ? g : pl.slabs;
    // With K <= 4096 and a CTA or more per tile, every tile is cut into the same number of parts
    // (the largest multiple of the tile count that fits): the longest part is no longer, no CTA
    // streams more than with the extra CTAs, and the HBM share of each CTA grows.  Measured on
    // GB300 (graph replays, weights L2-prefetched before the dependency wait): M = 16, K = 4096,
    // N = 12288 12.87 -> 11.89 us (192 CTAs), N = 8192 8.34 -> 8.16 (256), N = 2560 5.01 -> 4.92
    // (280), K = 2048, N = 4096 4.67 -> 4.51 (256); M = 32, N = 2560 6.96 -> 6.78.  With longer
    // tiles the extra CTAs win, their prefetch covering more of the stream before the wait
    // (K = 12288, N = 4096: 10.52 us at 304 CTAs against 10.75 at 256; K = 14336 11.65 against
    // 12.08), so K > 4096 keeps them.
    if (pl.kb <= 128 && gg >= pl.n_tiles) gg = (long long)pl.n_tiles * (gg / pl.n_tiles);
    pl.blocks = (int)gg;
  } else {
    if (blocks > pl.slabs) return W8A8_ERR_INVALID_ARG;
    pl.blocks = blocks;
  }
  // Two-element combine words when both fields and the arrival count fit: every partial sum of an
  // element is at most K * 2^14 in magnitude (|x|, |w| <= 128), so a signed field of f bits with
  // 2^(f-1) > K * 2^14 holds it, and the count needs 64 - 2f bits for the most CTAs sharing a tile.
  {
    const long long lim = (long long)K << 14;
    int bits = 0;
    while ((1ll << bits) <= lim) ++bits;
    const int f = bits + 1, count_bits = 64 - 2 * f;
    const GemmSplit sp = make_gemm_split(pl.n_tiles, pl.kb, pl.blocks, true);
    int most = 0;
    for (int t = 0; t < pl.n_tiles; ++t) {
      const int c = gemm_split_contributors(sp, t);
      most = c > most ? c : most;
    }
    pl.pack_f = (count_bits >= 1 && count_bits < 63 && (long long)most < (1ll << count_bits)) ? f : 0;
  }
  pl.threads = pl.blocks >= pl.n_tiles ? kThreadsNoCombine : kThreads;
  pl.split_unit = 1 << make_gemm_split(pl.n_tiles, pl.kb, pl.blocks, true).qs;
  pl.stage_slabs = kStageSlabs;
  pl.stages = gemm_stages(pl.nt8);
  pl.smem_bytes = gemm_smem_bytes(pl.nt8);
  // One 64-bit (arrival count, biased sum) word per output element of every tile.
  const size_t partials = (size_t)pl.n_tiles * kSubTiles * pl.nt8 * 4 * 32 * sizeof(unsigned long long);
  pl.partials_offset = kWsHeaderBytes;
  pl.workspace_bytes = kWsHeaderBytes + partials;
  *plan = pl;
  return W8A8_OK;
}

template <int NT8, int NS, bool kMulti>
static cudaError_t launch_gemm(const GemmParams& p, int blocks, int threads, cudaStream_t stream) {
  auto kern = w8a8_gemm_kernel<NT8, NS, kMulti>;
  const int smem = GemmLayout<NT8, NS>::kBytes;
  cudaError_t e = ensure_smem_attribute((const void*)kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  // Always a programmatic dependent of the work before it: before its dependency wait the kernel
  // reads or writes no global memory, only prefetches weight bytes into L2, unless W8A8_FLAG_PDL
  // allows the weight stream to start (p.pdl), so the overlap with the previous kernel's tail
  // needs nothing from the caller.  Measured on GB300
  // against plain launches (graph replays): gate_up M = 16 20.24 -> 19.42 us, M = 32 37.1 -> 33.6
  // us, the QKV-like shape 5.58 -> 4.65 us.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t gemm_launch(const GemmPlan& pl, const int8_t* x, const float* xs, const void* wp, const float* wsc,
                        void* out, int M, int K, int N, void* ws, bool pdl, cudaStream_t stream, int* acc, bool stall) {
  GemmParams p;
  // Activation tensor map: [M rows, K bytes], box of 128 bytes x 8*NT8 rows (rows >= M read as 0).
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {128u, (cuuint32_t)(8 * pl.nt8)};
  const cuuint32_t estr[2] = {1u, 1u};
  cudaError_t e = encode_tensor_map_2d(&p.xmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<int8_t*>(x), dims, strides,
                                       box, estr, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  p.wp = static_cast<const uint8_t*>(wp);
  p.x_scale = xs;
  p.w_scale = wsc;
  p.out = static_cast<uint16_t*>(out);
  p.status = static_cast<uint32_t*>(ws);
  p.tile_acc = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) + pl.partials_offset);
  p.M = M;
  p.K = K;
  p.N = N;
  p.KB = pl.kb;
  p.split = make_gemm_split(pl.n_tiles, pl.kb, pl.blocks, true);
  p.pack_f = pl.pack_f;
  p.pdl = pdl ? 1 : 0;
  p.acc_out = acc;
  p.debug_stall = stall ? 1 : 0;
  const bool multi = pl.threads == kThreads;
  switch (pl.nt8) {
    case 1: return multi ? launch_gemm<1, kStages1, true>(p, pl.blocks, pl.threads, stream)
                         : launch_gemm<1, kStages1, false>(p, pl.blocks, pl.threads, stream);
    case 2: return multi ? launch_gemm<2, kStages2, true>(p, pl.blocks, pl.threads, stream)
                         : launch_gemm<2, kStages2, false>(p, pl.blocks, pl.threads, stream);
    case 3: return multi ? launch_gemm<3, kStages3, true>(p, pl.blocks, pl.threads, stream)
                         : launch_gemm<3, kStages3, false>(p, pl.blocks, pl.threads, stream);
    default: return multi ? launch_gemm<4, kStages4, true>(p, pl.blocks, pl.threads, stream)
                          : launch_gemm<4, kStages4, false>(p, pl.blocks, pl.threads, stream);
  }
}

cudaError_t pack_launch(const int8_t* W, int K, int N, void* out, cudaStream_t stream) {
  const int KB = K / kKBlock;
  const long long tiles = (N + kTileRows - 1) / kTileRows;
  const long long chunks = tiles * KB * 4 * 32;
  long long grid = (chunks + 255) / 256;
  if (grid > 65535) grid = 65535;
  w8a8_pack_kernel<<<(unsigned)grid, 256, 0, stream>>>(W, K, N, KB, chunks, static_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace w8a8
