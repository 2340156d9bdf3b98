/*
 * w8a8.h - C ABI of the GB300 (sm_103a) small-M quantized weight GEMM library.
 *
 * Two operators of an LLM serving engine's decode and speculative-verify windows:
 *
 *  w8a8_gemm   x_q[M,K] int8 @ W[K,N] int8 -> int32, then * x_scale[M] * w_scale[N] -> bf16[M,N],
 *              M <= 128.  Defined by the operator line of "INT8 W8A8 GEMM - Decode (M <= 32) -
 *              gfx928 / SGLang TP4" (header paragraph); split-K with a fused last-arrival combine
 *              follows its section 1.1 (qkv recipe) and "Cross-shape rules that held".  M <= 32
 *              runs the decode arm; 32 < M <= 128 runs a second, staged arm on the tcgen05 tensor
 *              cores over the same packed weight (that page's section 3 keeps such an arm beside
 *              the decode one for the same (K, N)).
 *  q8_0_gemv   y[T,N] = x[T,K] (bf16) times Q8_0 weights (blocks of 32 int8 quants along K with one
 *              fp16 scale each), T <= 8, bf16 out.  Defined by "sycl: STRATA_HC_Q8=1 reads the Q8_0
 *              hyper-connection projections", section "What changed" (w = d * q, the split layout,
 *              fixed-order partial sums, last work-group combine).
 *  q8_0_gemv_rms  the same read with an RMS-norm prologue: y = rs[t] * (x * gamma) @ w (same page,
 *              same section: the down kernel's R' * w_norm staging with the sums of squares).
 *
 * Conventions for every entry point:
 *  - Data pointers are DEVICE pointers (cudaMalloc or equivalent) unless stated otherwise; the
 *    caller owns every buffer.  `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *  - Every argument check happens on the host before any launch.  A failed check launches
 *    nothing and returns a non-zero status; nothing is thrown and nothing is printed.
 *  - w8a8_gemm and q8_0_gemv do no host synchronisation, allocation or memset, so a call can be
 *    captured into a CUDA graph and replayed.  Each is one kernel launch, except w8a8_gemm with
 *    M > 32: two launches on the tcgen05 arm (the activations converted to fp16 into the
 *    workspace, then the GEMM as a programmatic dependent of that launch), or ceil(M / 32) decode
 *    launches when the automatic plan runs row chunks (see W8A8_FLAG_TENSOR_MEMORY_ARM).
 *  - A workspace is caller-owned device memory, at least 256-byte aligned, sized with the
 *    *_workspace_bytes queries and zeroed once with w8a8_workspace_init (outside any capture)
 *    before its first use.  Every call leaves it ready for the next one (each arrival counter is
 *    reset by the last arrival, and every accumulator returned to zero).  Calls that use the
 *    same workspace must not overlap in time (use one stream per workspace); one workspace may
 *    serve both operators in turn if it is sized for the larger of the two.
 *  - bf16 and fp16 values are passed as their 16-bit patterns (uint16_t storage).
 */
#ifndef W8A8_GB300_H
#define W8A8_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host status codes returned by every entry point. */
enum {
    W8A8_OK = 0,
    W8A8_ERR_INVALID_ARG = 1,         /* null pointer, M/T/K/N out of range, bad blocks count */
    W8A8_ERR_UNSUPPORTED_SHAPE = 2,   /* K % 32 != 0, N % 8 != 0 (w8a8) or K % 32 != 0 (q8_0) */
    W8A8_ERR_MISALIGNED = 3,          /* a pointer misses the alignment stated for it */
    W8A8_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the size query's answer */
    W8A8_ERR_CUDA = 5                 /* a CUDA runtime call failed; see w8a8_last_error() */
};

/* Device status bits, OR-ed into the first word of a workspace by a kernel that hit a fault
 * it could survive; read back with w8a8_workspace_status.  Both leave the outputs undefined. */
enum {
    W8A8_DEV_WAIT_TIMEOUT = 1u,       /* a pipeline wait exceeded its bound (about one second);
                                         the kernel abandoned the call and returned */
    W8A8_DEV_COUNTER_CORRUPT = 2u     /* an arrival counter held a value outside [0, arrivals):
                                         the workspace was not zeroed, or calls overlapped */
};

/* Launch flags of w8a8_gemm and q8_0_gemv. */
enum {
    /* Every w8a8_gemm decode launch (M <= 32, and the row chunks of larger M) and every q8_0_gemv
     * launch is a programmatic dependent of the work queued before it on the stream, flag or not:
     * its CTAs may become resident and set themselves up while the previous kernel finishes, and
     * read or write no global memory until that kernel has completed and its writes are visible.
     * Before that point they only prefetch their first weight bytes into L2, a hint that changes
     * no value any read returns.  This needs nothing from the caller and behaves as plain stream
     * order.
     * W8A8_FLAG_PDL (programmatic dependent launch with weight prefetch) also lets the kernel start
     * streaming the packed weight (W_packed, or q, d and gamma of q8_0_gemv) before that point;
     * every other input, the output and the workspace are still touched only after it.  The caller
     * guarantees that the weight buffers are not written by work still in flight on the stream
     * (weights are load-time constants: pack them, then synchronise once).  Consecutive calls then
     * overlap one call's weight prefetch with the previous call's tail, inside a CUDA graph as
     * well. */
    W8A8_FLAG_PDL = 1u,
    /* w8a8_gemm with 32 < M <= 128: always run the tcgen05 arm.  Without it the automatic plan
     * (blocks == 0) runs, whichever a cost model measured on GB300 predicts faster, either that
     * arm or the decode arm over consecutive chunks of at most 32 activation rows (one launch per
     * chunk, in stream order on the one workspace); an explicit blocks > 0 selects the tcgen05
     * arm as well.  Both give the same bits. */
    W8A8_FLAG_TENSOR_MEMORY_ARM = 2u,
    /* Test hook of the device fault path (w8a8_gemm and its variants only; not for production
     * calls).  One warp of the first CTA waits on a pipeline barrier that nothing completes, with a
     * bound of a few milliseconds instead of the usual second.  The wait runs out, the kernel
     * records W8A8_DEV_WAIT_TIMEOUT in the workspace status word, and every CTA returns: the rest
     * of that CTA gives up at its next wait, after the copies it issued have landed and the tensor
     * memory it holds is freed.  The host call itself returns W8A8_OK; the output is undefined and
     * the workspace must be zeroed again (w8a8_workspace_init) before its next use.  No GPU fault
     * and no hang is involved: it exercises the same bounded-wait exit that a real timeout takes. */
    W8A8_FLAG_TEST_STALL = 0x100u
};

/* Library version (major * 10000 + minor * 100 + patch). */
int w8a8_version(void);

/* Static text for a host status code. */
const char* w8a8_status_string(int status);

/* Text of the last CUDA error seen by this thread inside the library ("" if none). */
const char* w8a8_last_error(void);

/* -------------------------------------------------------------------------------------------
 * Workspaces
 * ----------------------------------------------------------------------------------------- */

/* Zero a workspace (one cudaMemsetAsync of ws_bytes on `stream`).  Call once after allocating
 * it, before any w8a8_gemm / q8_0_gemv call that uses it and outside any stream capture; the
 * qkv recipe of section 1.1 of the W8A8 page keeps its counters in the workspace and clears them
 * with one async memset before the first launch.  Errors: INVALID_ARG (ws NULL or ws_bytes 0),
 * MISALIGNED (ws not 256-byte aligned), CUDA. */
int w8a8_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Read the device status word of a workspace into *status (0 = no device fault recorded), and
 * clear it.  Synchronises `stream` (a host read): not for use inside a capture. */
int w8a8_workspace_status(void* ws, size_t ws_bytes, void* stream, uint32_t* status);

/* -------------------------------------------------------------------------------------------
 * W8A8 decode GEMM
 * ----------------------------------------------------------------------------------------- */

/* Bytes of the packed weight for a [K,N] int8 W: 64 * ceil(N/64) * K. */
size_t w8a8_packed_weight_bytes(int K, int N);

/* Workspace bytes that w8a8_gemm needs for every M in [1, M_max] (M_max <= 128) at this (K, N)
 * and `blocks` (0 = the automatic plan, whose CTA count follows the current device's SM count).
 * Returns 0 for arguments w8a8_gemm would reject.  Layout: a 256-byte header (status word first),
 * then, for M <= 32, one 64-bit accumulator word per output element of every 64-row tile (zero
 * between calls); for M > 32, one 32-bit arrival counter per 128-row tile (padded to 256 bytes)
 * and one int32 sum per (tile, activation row < 128, tile row), both zero between calls, then the
 * call's activations as fp16 [M][K] (overwritten by every call).  The regions sit at offsets that
 * do not depend on M, so calls of any M in [1, M_max] may share one workspace in turn. */
size_t w8a8_workspace_bytes(int M_max, int K, int N, int blocks);

/* Pack W once, at load time and outside any timed region or capture (section 1.1 of the W8A8
 * page, third cross-shape rule: the cold once-read weight is packed into the fragment's layout
 * so that every fragment is one contiguous vector read).
 *
 *  W         [K,N] int8, row-major (W[k][n] at k*N + n), device memory.
 *  W_packed  device buffer of w8a8_packed_weight_bytes(K, N) bytes, 16-byte aligned.  Layout,
 *            with Np = 64*ceil(N/64), KB = K/32, g = lane/4, c = lane%4, w = j/4, b = j%4:
 *              byte ((((t*KB + kb)*4 + s)*32 + lane)*16 + j)  for t < Np/64, kb < KB, s < 4,
 *              lane < 32, j < 16 holds  W[k][n] XOR 0x80  (offset binary; 0x80 for n >= N) with
 *              n = 64t + 16s + g + 8(w%2),  k = 32kb + 8c + 4(w/2) + b.
 *            So each 64-row tile t is one contiguous run of KB 2-KiB slabs, and a CTA whose share
 *            of the work is a run of slabs streams one contiguous byte range.
 *  ws        optional workspace; if not NULL it is zeroed as by w8a8_workspace_init.
 *  Requires K % 32 == 0, 1 <= K <= 65536, 1 <= N <= 1048576, N % 8 == 0.
 *  Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA. */
int w8a8_pack_weights(const int8_t* W, int K, int N, void* W_packed, void* ws, size_t ws_bytes,
                      void* stream);

/* out[m][n] = bf16_rne( ((float)acc[m][n] * x_scale[m]) * w_scale[n] ),
 * acc[m][n] = sum_k x_q[m][k] * W[k][n] in exact int32.
 *
 *  x_q      [M,K] int8 row-major, 16-byte aligned.     x_scale  [M] fp32.
 *  W_packed from w8a8_pack_weights(W, K, N, ...).      w_scale  [N] fp32.
 *  out      [M,N] bf16 row-major (uint16_t storage), 16-byte aligned; rows m >= M and columns
 *           n >= N are never written.
 *  M in [1, 128]; K % 32 == 0; N % 8 == 0 (same limits as the pack).
 *  blocks   number of CTAs that share the T = ceil(N/64) tiles x KB = K/32 slabs of 2 KiB
 *           (split-K generalised; every cut lies on a 32-aligned k).  With blocks >= T each tile
 *           is cut into c + 1 (the first blocks % T tiles) or c = blocks / T contiguous parts of
 *           equal length to within one slab, one per CTA, so no CTA spans two tiles; with
 *           blocks < T the tiles are laid end to end and CTA i takes a contiguous run of
 *           ceil or floor(T KB / (u blocks)) units of u slabs (the longer runs first), u being
 *           the plan's split_unit (1 or 4; see w8a8_plan_t).  0 = automatic: twice the SM
 *           count, at most one CTA per slab; for K <= 4096 with that count >= T, rounded down
 *           to a multiple of T so that every tile is cut into the same number of parts.  Must not
 *           exceed the number of slabs.
 *           For M > 32 the same rule applies to T = ceil(N/128) tiles of 128 rows (two packed
 *           tiles each) x KB units of 32 k, with one CTA per SM by default.
 *  flags    0, W8A8_FLAG_PDL and/or W8A8_FLAG_TENSOR_MEMORY_ARM (W8A8_FLAG_TEST_STALL for tests
 *           of the fault path); any other bit is INVALID_ARG.
 *  ws       workspace of at least w8a8_workspace_bytes(M, K, N, blocks) bytes.
 *  The int32 sums are exact (the result does not depend on `blocks`), and the epilogue order is
 *  fixed, so the output is bit-identical for every `blocks` and every replay.
 *  Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA. */
int w8a8_gemm(const int8_t* x_q, const float* x_scale, const void* W_packed, const float* w_scale,
              void* out, int M, int K, int N, int blocks, unsigned flags, void* ws, size_t ws_bytes,
              void* stream);

/* The same call as w8a8_gemm, which in addition stores the exact int32 sums
 *   acc[m][n] = sum_k x_q[m][k] * W[k][n]
 * that its epilogue scales, into `acc` ([M,N] int32 row-major, 4-byte aligned, device memory;
 * rows m >= M and columns n >= N are never written).  The W8A8 page's cross-shape rules make the
 * int32 accumulation exact and its outputs bit-identical across splits; this entry point exposes
 * the accumulators so that they can be checked against a reference bit for bit, not only through
 * the bf16 rounding.  The same kernel runs, with one more store per output element.
 * Errors: those of w8a8_gemm, and INVALID_ARG for a NULL acc, MISALIGNED for a misaligned one. */
int w8a8_gemm_acc(const int8_t* x_q, const float* x_scale, const void* W_packed, const float* w_scale,
                  void* out, int32_t* acc, int M, int K, int N, int blocks, unsigned flags, void* ws,
                  size_t ws_bytes, void* stream);

/* Launch plan of a w8a8_gemm call (host-only query; launches nothing). */
typedef struct {
    int n8_tiles;          /* column tiles of 8 covering M: 1..4, or 8 / 16 (MMA N = 64 / 128) */
    int n_tiles;           /* tiles of N (tile_rows rows each) */
    int k_blocks;          /* K / 32 */
    long long slabs;       /* n_tiles * k_blocks: the split's units (32 k of one tile each) */
    int blocks;            /* CTAs launched */
    int threads;           /* threads per CTA */
    int stage_slabs;       /* slabs per pipeline stage */
    int stages;            /* pipeline depth */
    size_t smem_bytes;     /* dynamic shared memory per CTA */
    size_t workspace_bytes;/* workspace this call needs */
    int combine_pack_bits; /* split-tile combine: 0 = one output element per 64-bit workspace word,
                              f > 0 = two elements per word in f-bit fields plus a 64 - 2f bit
                              arrival count (chosen when both fit; halves the atomics) */
    int tile_rows;         /* weight rows per tile: 64 (M <= 32) or 128 (M > 32) */
    int tensor_memory;     /* 1: the tcgen05 arm (accumulators in tensor memory), 0: decode arm */
    int row_chunks;        /* decode launches per call: 1, or ceil(M / 32) when the automatic plan
                              runs 32 < M <= 128 as row chunks (the other fields describe the plan
                              of a 32-row chunk) */
    int split_unit;        /* slabs per unit of a run split with blocks < n_tiles: 1, or 4 for the
                              decode arm when K % 128 == 0 and runs of whole 4-slab units make the
                              longest run at most 3 % longer (every run then starts on an 8 KiB
                              boundary of the packed weight) */
} w8a8_plan_t;

int w8a8_plan(int M, int K, int N, int blocks, w8a8_plan_t* plan);

/* The plan of a w8a8_gemm call made with `flags` (W8A8_FLAG_TENSOR_MEMORY_ARM changes the plan of
 * 32 < M <= 128; the other flags do not).  Host-only. */
int w8a8_plan_flags(int M, int K, int N, int blocks, unsigned flags, w8a8_plan_t* plan);

/* The slab runs of a plan (the split described at w8a8_gemm's `blocks`): bounds[i] = first
 * slab of CTA i, bounds[blocks] = total slabs (slab u covers tile u / KB, k in
 * [32 (u % KB), 32 (u % KB) + 32)).  n_bounds must be blocks + 1.  Host-only. */
int w8a8_split_bounds(int K, int N, int blocks, long long* bounds, int n_bounds);

/* The same for the plan of an M-row call (M > 32: units of 32 k of a 128-row tile). */
int w8a8_split_bounds_m(int M, int K, int N, int blocks, long long* bounds, int n_bounds);

/* W8A8 GEMM (both arms) that allocates nothing and takes no workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot provide device memory, such as a
 * plugin that sees only the input and output pointers its host engine hands it, or a request path
 * that must not call cudaMalloc (which can synchronise the device and stall other streams).
 *
 * Arguments, limits and result are those of w8a8_gemm, without ws / ws_bytes; flags as for
 * w8a8_gemm.  The workspace is a 16 MiB area inside this library's device memory (a file-scope
 * __device__ array, held on every device that loads the library until the process exits); a shape
 * whose w8a8_workspace_bytes(M, K, N, blocks) exceeds 16 MiB returns W8A8_ERR_WORKSPACE_TOO_SMALL.
 * Each call clears the part of the area its kernel needs zeroed (one cudaMemsetAsync on `stream`)
 * and then launches the kernel; it calls no allocating routine.
 *
 * The first call in a CUDA context looks up the area's device address (cudaGetSymbolAddress, in
 * that context) and caches it per context; make that first call before any stream capture.  A
 * context created later (another context on the device, or the primary context again after
 * cudaDeviceReset) gets its own look-up on its first call.  All calls in a context share the one
 * area, so calls whose kernels can overlap on the GPU (on different streams without ordering
 * between them) race on it and give undefined results.
 *
 * Device faults (W8A8_DEV_*) are OR-ed into the area's status word, which no call clears: read it
 * with w8a8_gemm_no_alloc_status. */
int w8a8_gemm_no_alloc(const int8_t* x_q, const float* x_scale, const void* W_packed,
                       const float* w_scale, void* out, int M, int K, int N, int blocks,
                       unsigned flags, void* stream);

/* Read the device status word of w8a8_gemm_no_alloc's area in the current context into *status
 * (0 = no device fault recorded since the last read; otherwise W8A8_DEV_* bits of any call since
 * then), and clear it.  Synchronises `stream` (a host read): not for use inside a capture.  Errors:
 * INVALID_ARG (status NULL), CUDA. */
int w8a8_gemm_no_alloc_status(void* stream, uint32_t* status);

/* -------------------------------------------------------------------------------------------
 * Q8_0 weight GEMV (verify window)
 * ----------------------------------------------------------------------------------------- */

/* Workspace bytes that q8_0_gemv needs for every T in [1, T_max] at (K, N). */
size_t q8_0_workspace_bytes(int T_max, int K, int N);

/* y[t][n] = bf16_rne( sum_k x[t][k] * (d[n][k/32] * q[n][k]) ), summed in fp32 in a fixed order
 * (bit-identical across replays).
 *
 *  x   [T,K] bf16 row-major, 16-byte aligned.
 *  q   [N,K] int8 row-major: the quants of the split layout, 16-byte aligned.
 *  d   [N,K/32] fp16 row-major: the block scales of the split layout (scale of q[n][32b..32b+31]
 *      is d[n][b]), 2-byte aligned.
 *  y   [T,N] bf16 row-major, 2-byte aligned; rows t >= T are never written.
 *  T in [1, 8]; K % 32 == 0, 32 <= K <= 65536; 1 <= N <= 1048576.
 *  flags 0 or W8A8_FLAG_PDL; any other bit is INVALID_ARG.
 *  Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA. */
int q8_0_gemv(const void* x, const int8_t* q, const void* d, void* y, int T, int K, int N,
              unsigned flags, void* ws, size_t ws_bytes, void* stream);

/* The Q8_0 read with an RMS-norm prologue:
 *   y[t][n] = bf16_rne( rs[t] * sum_k bf16(x[t][k] * gamma[k]) * (d[n][k/32] * q[n][k]) ),
 *   rs[t]   = 1 / sqrt(sum_k x[t][k]^2 / K + eps),
 * the generic form of "sycl: STRATA_HC_Q8=1 reads the Q8_0 hyper-connection projections", section
 * "What changed" (the down kernel stages R' * w_norm unscaled with the rows' sums of squares, and
 * the last work-group to arrive applies rs per stream).  The product x * gamma is exact in fp32 and
 * rounded once to bf16 (the MMA's operand); the sums of squares are fp32 in a fixed order; rs is
 * IEEE division and square root.  Replays are bit-identical.
 *  gamma  [K] bf16 (the norm weight), 16-byte aligned; read before the dependency wait under
 *         W8A8_FLAG_PDL, like q and d (a weight).
 *  eps    finite and >= 0, else INVALID_ARG.
 *  Everything else, the workspace (q8_0_workspace_bytes) and the errors as q8_0_gemv. */
int q8_0_gemv_rms(const void* x, const void* gamma, float eps, const int8_t* q, const void* d,
                  void* y, int T, int K, int N, unsigned flags, void* ws, size_t ws_bytes,
                  void* stream);

/* ---------------------------------------------------------------------------------------------
 * Quantisation around the operators (outside the timed GEMM / read).  Sources: the Q8_0 page
 * ("sycl: STRATA_HC_Q8=1 reads the Q8_0 hyper-connection projections", section "What changed",
 * the loader bullet: d = amax / 127 stored as fp16, q = round(x / d), split layout); the W8A8
 * page's operator line (x_q int8 with x_scale[M,1]; quantisation is outside the timed region).
 * Readings: amax per 32-value block (Q8_0) or per row (activations); x is divided by the float32
 * scale; round = C roundf (halves away from zero); an all-zero block or row gets scale 0 and
 * quants 0; inputs are finite.  Division and fp16 conversion round to nearest even, so results
 * are bit-identical to a scalar IEEE evaluation.  All pointers are device pointers; each call is
 * one kernel launch on `stream`, graph-capture safe, with every check done before it.
 * ------------------------------------------------------------------------------------------- */

/* x [M,K] bf16 row-major (16-byte aligned) -> x_q [M,K] int8 (8-byte aligned) and
 * x_scale [M] fp32: x_scale[m] = max_k |x[m][k]| / 127, x_q[m][k] = roundf(x[m][k] / x_scale[m]).
 * 1 <= M <= 2^20, 8 <= K <= 65536, K % 8 == 0.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE,
 * MISALIGNED, CUDA.
 * The kernel lets a programmatic dependent launched after it on the stream start at once
 * (griddepcontrol.launch_dependents), so that a following w8a8_gemm prefetches its weights while
 * it runs.  A dependent kernel of the caller's own must wait for the grid
 * (griddepcontrol.wait or cudaGridDependencySynchronize) before it reads x_q or x_scale, as
 * every kernel of this library does. */
int w8a8_quantize_activations(const void* x, int8_t* x_q, float* x_scale, int M, int K, void* stream);

/* Q8_0 from BF16 weights: w [N,K] bf16 row-major (16-byte aligned) -> the split layout of
 * q8_0_gemv, q [N,K] int8 (8-byte aligned) and d [N,K/32] fp16 (2-byte aligned), per block of 32
 * along K: d = fp16_rn(amax / 127), q = roundf(w / (amax / 127)).  K % 32 == 0, 32 <= K <= 65536,
 * 1 <= N <= 2^20.  Errors as above. */
int q8_0_quantize(const void* w, int8_t* q, void* d, int K, int N, void* stream);

/* ggml-style Q8_0 rows (per block: the fp16 scale little-endian, then its 32 quants; 34 bytes;
 * blocks [N][K/32], 2-byte aligned) -> the split layout (q [N,K] 16-byte aligned, d [N,K/32]), and
 * back.  The same bytes, reordered.  Limits and errors as for q8_0_quantize. */
int q8_0_split_from_blocks(const void* blocks, int8_t* q, void* d, int K, int N, void* stream);
int q8_0_blocks_from_split(const int8_t* q, const void* d, void* blocks, int K, int N, void* stream);

/* Measurement helper (not part of either operator): reads `bytes` (rounded down to a multiple of
 * 16) of device memory at `buf` once with 16-byte vector loads, on 2 x SM-count CTAs of 512
 * threads, and discards the data (a 64-bit device word at `sink` is written only in a case that
 * real data practically never produce).  Timed over a buffer larger than L2 it gives the
 * achievable HBM read rate, the ceiling for the weight stream.  buf 16-byte aligned, sink 8-byte
 * aligned.  Errors: INVALID_ARG, MISALIGNED, CUDA. */
int w8a8_read_probe(const void* buf, size_t bytes, void* sink, void* stream);

/* Measurement helper (not part of either operator): the tensor-pipe rate of the two register-fed
 * MMA forms an int8 product can take, for the caller to time.  kind 0: mma.sync m16n8k16 with fp16
 * operands and fp32 accumulation (4096 flops per MMA; the form the decode kernel uses, after its
 * exact int8 -> fp16 conversion); kind 1: mma.sync m16n8k32 with int8 operands and int32
 * accumulation (8192 int ops per MMA).  One launch of 2 x SM-count CTAs of 256 threads; every warp
 * issues iters x 8 independent MMAs, so one call performs 2 x SMs x 8 x iters x 8 MMAs.  sink: an
 * 8-byte aligned device word written only in a case real runs practically never produce.
 * iters in [1, 2^24].  Errors: INVALID_ARG, MISALIGNED, CUDA. */
int w8a8_mma_rate_probe(int kind, int iters, void* sink, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_GB300_H */
