/*
 * Oracle for the small-M quantized weight GEMMs: plain, slow, obviously correct
 * CPU code.  TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
 * benchmark's CPU-baseline leg use it; the library's compute path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (web pages; section names as printed there):
 *  [W8A8] "INT8 W8A8 GEMM - Decode (M <= 32) - gfx928 / SGLang TP4", operator line:
 *         x_q[M,K] int8 @ W[K,N] int8 -> int32 -> * x_scale[M,1] * weight_scale[N,1].T -> bf16[M,N].
 *         Section 1.1, "Cross-shape rules that held": int32 accumulation that is k-ascending per
 *         split, then an ascending sum over splits; "[0,K) exactly once".
 *  [Q8_0] "sycl: STRATA_HC_Q8=1 reads the Q8_0 hyper-connection projections", section
 *         "What changed": Q8_0 weights as blocks of 32 int8 quants with one fp16 scale,
 *         dequantised as w = d * q; the split layout (every row's quants row-major, then every
 *         row's fp16 scales); the parity test's FP64 reference computed from the very Q8_0
 *         bytes the kernel reads.
 *
 * Readings where the pages leave a step open (the plainest reading the rest of the pages support):
 *  - The W8A8 epilogue is (float(acc) * x_scale[m]) * w_scale[n], each step an IEEE fp32
 *    multiply rounded to nearest even, then rounded to nearest even into bfloat16.  The pages
 *    only say "scales ... bf16"; the library's interface defines this order, x_scale first.
 *  - Q8_0 blocks run along K inside each weight row n; d has shape [N, K/32].
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC (see build.py).
 * Every float operation below is a single IEEE operation: no contraction, no x87.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ---------------------------------------------------------------------------------------
 * bfloat16 / float16 scalars, written from the IEEE-754 definitions.
 * ------------------------------------------------------------------------------------- */

/* float32 -> bfloat16 bits, round to nearest, ties to even.  bfloat16 keeps the top 16 bits
 * of the float32 encoding; the discarded low half decides the rounding: above 0x8000 rounds
 * up, below rounds down, exactly 0x8000 rounds to the even upper half.  NaN inputs keep a
 * quiet NaN (never reached by the W8A8 epilogue, whose values are finite). */
uint16_t oracle_bf16_from_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;               /* a carry into the exponent is the correct rounding */
    return (uint16_t)upper;
}

double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* IEEE binary16 -> double: sign, 5-bit exponent (bias 15), 10-bit fraction. */
double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)frac, -24);                  /* subnormal: frac * 2^-14 * 2^-10 */
    else if (e == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), e - 25);      /* (1 + frac/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* ---------------------------------------------------------------------------------------
 * W8A8 decode GEMM  [W8A8] operator line.
 * ------------------------------------------------------------------------------------- */

/* acc[m][n] = sum_{k=0}^{K-1} x_q[m][k] * W[k][n], summed in int64 and then checked to fit
 * int32 (the operator's accumulator type).  x_q is [M,K] row-major, W is [K,N] row-major.
 * Returns 0, or -1 if some sum leaves the int32 range. */
int oracle_w8a8_acc(const int8_t* x_q, const int8_t* W, int M, int K, int N, int32_t* acc) {
    int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    int rc = 0;
    if (!row) return -2;
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) row[n] = 0;
        for (int k = 0; k < K; ++k) {
            int64_t xv = x_q[(size_t)m * K + k];
            const int8_t* wk = W + (size_t)k * N;
            for (int n = 0; n < N; ++n) row[n] += xv * (int64_t)wk[n];
        }
        for (int n = 0; n < N; ++n) {
            if (row[n] > INT32_MAX || row[n] < INT32_MIN) rc = -1;
            acc[(size_t)m * N + n] = (int32_t)row[n];
        }
    }
    free(row);
    return rc;
}

/* The same sums taken the way a split-K kernel takes them ([W8A8] section 1.1): the K range is
 * cut at bounds[0]=0 < bounds[1] < ... < bounds[parts]=K; each slice is summed k-ascending in
 * int32, and the slice sums are added in ascending slice order in int32.  Returns -1 if the
 * bounds do not cover [0,K) exactly once in ascending order. */
int oracle_w8a8_acc_split(const int8_t* x_q, const int8_t* W, int M, int K, int N,
                          const int* bounds, int parts, int32_t* acc) {
    if (parts < 1 || bounds[0] != 0 || bounds[parts] != K) return -1;
    for (int p = 0; p < parts; ++p)
        if (bounds[p + 1] < bounds[p]) return -1;
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            int32_t total = 0;
            for (int p = 0; p < parts; ++p) {
                int32_t slice = 0;
                for (int k = bounds[p]; k < bounds[p + 1]; ++k)
                    slice += (int32_t)x_q[(size_t)m * K + k] * (int32_t)W[(size_t)k * N + n];
                total += slice;
            }
            acc[(size_t)m * N + n] = total;
        }
    }
    return 0;
}

/* out[m][n] = bf16_rne( fp32( fp32(float(acc[m][n]) * x_scale[m]) * w_scale[n] ) ).
 * (float)acc is the C conversion, which rounds to nearest even for |acc| > 2^24. */
void oracle_w8a8_epilogue(const int32_t* acc, const float* x_scale, const float* w_scale,
                          int M, int N, uint16_t* out) {
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            float f = (float)acc[(size_t)m * N + n];
            volatile float a = f * x_scale[m];       /* volatile: keep two separate roundings */
            volatile float b = a * w_scale[n];
            out[(size_t)m * N + n] = oracle_bf16_from_f32(b);
        }
    }
}

/* Whole operator: accumulate, then the scale / bf16 epilogue.  acc may be NULL. */
int oracle_w8a8_gemm(const int8_t* x_q, const float* x_scale, const int8_t* W, const float* w_scale,
                     int M, int K, int N, uint16_t* out, int32_t* acc) {
    int32_t* a = acc ? acc : (int32_t*)malloc(sizeof(int32_t) * (size_t)M * (size_t)N + 4);
    if (!a) return -2;
    int rc = oracle_w8a8_acc(x_q, W, M, K, N, a);
    oracle_w8a8_epilogue(a, x_scale, w_scale, M, N, out);
    if (!acc) free(a);
    return rc;
}

/* ---------------------------------------------------------------------------------------
 * Q8_0 weight GEMV  [Q8_0] section "What changed".
 * ------------------------------------------------------------------------------------- */

/* y[t][n] = sum_k x[t][k] * (d[n][k/32] * q[n][k]) in double, from the very bf16 / fp16 /
 * int8 bytes the kernel reads.  x: bf16 bits [T,K]; q: int8 [N,K]; d: fp16 bits [N,K/32]. */
void oracle_q8_0_gemv(const uint16_t* x, const int8_t* q, const uint16_t* d,
                      int T, int K, int N, double* y) {
    int nb = K / 32;
    for (int t = 0; t < T; ++t) {
        for (int n = 0; n < N; ++n) {
            double s = 0.0;
            for (int k = 0; k < K; ++k) {
                double w = oracle_f16_to_f64(d[(size_t)n * nb + k / 32]) * (double)q[(size_t)n * K + k];
                s += oracle_bf16_to_f64(x[(size_t)t * K + k]) * w;
            }
            y[(size_t)t * N + n] = s;
        }
    }
}

/* Euclidean norms used by the per-output error bound: xnorm[t] = ||x_t||_2 and
 * wnorm[n] = ||w_n||_2 with w_n the dequantised weight row (w = d * q). */
void oracle_q8_0_norms(const uint16_t* x, const int8_t* q, const uint16_t* d,
                       int T, int K, int N, double* xnorm, double* wnorm) {
    int nb = K / 32;
    for (int t = 0; t < T; ++t) {
        double s = 0.0;
        for (int k = 0; k < K; ++k) {
            double v = oracle_bf16_to_f64(x[(size_t)t * K + k]);
            s += v * v;
        }
        xnorm[t] = sqrt(s);
    }
    for (int n = 0; n < N; ++n) {
        double s = 0.0;
        for (int k = 0; k < K; ++k) {
            double w = oracle_f16_to_f64(d[(size_t)n * nb + k / 32]) * (double)q[(size_t)n * K + k];
            s += w * w;
        }
        wnorm[n] = sqrt(s);
    }
}

/* Q8_0 read with an RMS-norm prologue.  [Q8_0] section "What changed": the down kernel stages
 * R' * w_norm unscaled together with the sums of squares of the rows, and the last work-group to
 * arrive applies rs per stream; the page does not define rs.  Generic reading: rs[t] is the inverse
 * root mean square of x's row t, 1 / sqrt(sum_k x[t][k]^2 / K + eps), and
 *   y[t][n] = rs[t] * sum_k (x[t][k] * g[k]) * (d[n][k/32] * q[n][k]),
 * all in double from the very bf16 / fp16 / int8 bytes the kernel reads.  x: bf16 bits [T,K];
 * g: bf16 bits [K] (w_norm); q, d as in oracle_q8_0_gemv; rs: out [T], may be NULL. */
void oracle_q8_0_rms_gemv(const uint16_t* x, const uint16_t* g, double eps, const int8_t* q,
                          const uint16_t* d, int T, int K, int N, double* y, double* rs) {
    int nb = K / 32;
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int k = 0; k < K; ++k) {
            double v = oracle_bf16_to_f64(x[(size_t)t * K + k]);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / (double)K + eps);
        if (rs) rs[t] = r;
        for (int n = 0; n < N; ++n) {
            double s = 0.0;
            for (int k = 0; k < K; ++k) {
                double xg = oracle_bf16_to_f64(x[(size_t)t * K + k]) * oracle_bf16_to_f64(g[k]);
                double w = oracle_f16_to_f64(d[(size_t)n * nb + k / 32]) * (double)q[(size_t)n * K + k];
                s += xg * w;
            }
            y[(size_t)t * N + n] = r * s;
        }
    }
}

/* xgnorm[t] = ||x_t * g||_2 (elementwise product), for the per-output error bound of the
 * RMS-norm read. */
void oracle_q8_0_rms_xg_norms(const uint16_t* x, const uint16_t* g, int T, int K, double* xgnorm) {
    for (int t = 0; t < T; ++t) {
        double s = 0.0;
        for (int k = 0; k < K; ++k) {
            double v = oracle_bf16_to_f64(x[(size_t)t * K + k]) * oracle_bf16_to_f64(g[k]);
            s += v * v;
        }
        xgnorm[t] = sqrt(s);
    }
}

/* ggml-style interleaved Q8_0 rows (per block: fp16 scale, then 32 int8 quants; 34 bytes)
 * -> the split layout (all quants [N][K], then all scales [N][K/32]).  [Q8_0] "What changed":
 * "the same bytes as ggml's 34-byte blocks, reordered". */
void oracle_q8_0_split_from_blocks(const uint8_t* blocks, int K, int N, int8_t* q, uint16_t* d) {
    int nb = K / 32;
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < nb; ++b) {
            const uint8_t* blk = blocks + ((size_t)n * nb + b) * 34;
            d[(size_t)n * nb + b] = (uint16_t)(blk[0] | (blk[1] << 8));
            for (int j = 0; j < 32; ++j) q[(size_t)n * K + (size_t)b * 32 + j] = (int8_t)blk[2 + j];
        }
    }
}

/* ---------------------------------------------------------------------------------------
 * Packed weight layout of w8a8_pack_weights, written out from its documented definition
 * (the library header states it; [W8A8] section 1.1 asks for the cold weight to be packed
 * once, outside the timed region, into the fragment's layout).
 *
 *   N is padded to Np = 64 * ceil(N / 64); KB = K / 32.
 *   byte (t, kb, s, lane, j), t < Np/64, kb < KB, s < 4, lane < 32, j < 16, sits at
 *     ((((t * KB + kb) * 4 + s) * 32 + lane) * 16 + j)
 *   and holds W[k][n] XOR 0x80 (offset binary), or 0x80 for a padding row n >= N, with
 *     g = lane / 4, c = lane % 4, w = j / 4, b = j % 4,
 *     n = 64 t + 16 s + g + 8 (w % 2),   k = 32 kb + 8 c + 4 (w / 2) + b.
 * ------------------------------------------------------------------------------------- */
size_t oracle_w8a8_packed_bytes(int K, int N) {
    size_t np = (size_t)((N + 63) / 64) * 64;
    return np * (size_t)K;
}

void oracle_w8a8_pack(const int8_t* W, int K, int N, uint8_t* packed) {
    int KB = K / 32;
    int tiles = (N + 63) / 64;
    for (int t = 0; t < tiles; ++t)
        for (int kb = 0; kb < KB; ++kb)
            for (int s = 0; s < 4; ++s)
                for (int lane = 0; lane < 32; ++lane)
                    for (int j = 0; j < 16; ++j) {
                        int g = lane / 4, c = lane % 4, w = j / 4, b = j % 4;
                        int n = 64 * t + 16 * s + g + 8 * (w % 2);
                        int k = 32 * kb + 8 * c + 4 * (w / 2) + b;
                        size_t off = ((((size_t)t * KB + kb) * 4 + s) * 32 + lane) * 16 + j;
                        packed[off] = n < N ? (uint8_t)(((uint8_t)W[(size_t)k * N + n]) ^ 0x80u) : 0x80u;
                    }
}

/* ---------------------------------------------------------------------------------------
 * Load-time and input-side quantisation (the rows after the hot path).
 * ------------------------------------------------------------------------------------- */

/* bfloat16 bits -> float32: the bfloat16 encoding is the top half of the float32 one. */
static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* float32 -> IEEE half bits, round to nearest, ties to even, from the two encodings.  A half
 * has 10 stored mantissa bits and exponent bias 15: normal halves cover [2^-14, 65504], the
 * subnormals are multiples of 2^-24 below 2^-14, and magnitudes from 65520 (halfway between
 * 65504 and 2^16) round to infinity. */
uint16_t oracle_f16_from_f32(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    const uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);   /* NaN */
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);  /* >= 65520: infinity */
    if (ax < 0x38800000u) {                                   /* below 2^-14: subnormal or zero */
        const uint32_t e = ax >> 23;
        if (e < 102) return sign;                              /* below 2^-25 (ties at 2^-25 go to 0) */
        const uint32_t m = (ax & 0x7FFFFFu) | 0x800000u;       /* value = m * 2^(e - 150) */
        const uint32_t shift = 126 - e;                        /* in units of 2^-24: m >> shift */
        uint32_t r = m >> shift;
        const uint32_t rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (r & 1u))) ++r;
        return (uint16_t)(sign | r);
    }
    const uint32_t rebased = ax - 0x38000000u;                 /* exponent bias 127 -> 15 */
    uint32_t r = rebased >> 13;
    const uint32_t rem = rebased & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) ++r;    /* a carry moves into the exponent */
    return (uint16_t)(sign | r);
}

/* Q8_0 quantisation of BF16 weights at load.  [Q8_0] "What changed", the loader bullet: a BF16
 * tensor is quantised on the host with ggml's rounding, d = amax / 127 stored as fp16 and
 * q = round(x / d), then uploaded in the split layout.  Readings where the pages are silent:
 * amax is taken over the 32 values of a block (the block is Q8_0's unit); the d that divides x
 * is the float32 quotient amax / 127, before it is stored as fp16; round is C's roundf (halves
 * away from zero); a block whose amax is 0 gets d = 0 and q = 0.
 *   w [N, K] bf16 bits, row-major -> q [N, K] int8, d [N, K / 32] fp16 bits. */
void oracle_q8_0_quantize(const uint16_t* w, int K, int N, int8_t* q, uint16_t* d) {
    const int nb = K / 32;
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < nb; ++b) {
            const uint16_t* blk = w + (size_t)n * K + (size_t)b * 32;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                const float a = fabsf(bf16_to_f32(blk[j]));
                if (a > amax) amax = a;
            }
            const float dd = amax / 127.0f;
            d[(size_t)n * nb + b] = oracle_f16_from_f32(dd);
            for (int j = 0; j < 32; ++j)
                q[(size_t)n * K + (size_t)b * 32 + j] = dd == 0.0f ? 0 : (int8_t)roundf(bf16_to_f32(blk[j]) / dd);
        }
    }
}

/* Per-row symmetric int8 quantisation of bf16 activations, the input side of the W8A8 operator.
 * [W8A8] operator line: x_q[M,K] int8 with x_scale[M,1], and the timed region "excludes
 * quantization" - the pages fix the scale's shape but not how it is computed.  Reading: the
 * Q8_0 loader's convention with one block per row, x_scale[m] = amax_m / 127 (float32) and
 * x_q[m][k] = roundf(x[m][k] / x_scale[m]), 0 for a row whose amax is 0.
 *   x [M, K] bf16 bits, row-major -> x_q [M, K] int8, x_scale [M] float32. */
void oracle_w8a8_quantize_rows(const uint16_t* x, int M, int K, int8_t* x_q, float* x_scale) {
    for (int m = 0; m < M; ++m) {
        const uint16_t* row = x + (size_t)m * K;
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            const float a = fabsf(bf16_to_f32(row[k]));
            if (a > amax) amax = a;
        }
        const float s = amax / 127.0f;
        x_scale[m] = s;
        for (int k = 0; k < K; ++k)
            x_q[(size_t)m * K + k] = s == 0.0f ? 0 : (int8_t)roundf(bf16_to_f32(row[k]) / s);
    }
}

/* The split layout -> ggml-style interleaved blocks (the inverse of oracle_q8_0_split_from_blocks):
 * per block the fp16 scale (little-endian), then its 32 quants; 34 bytes. */
void oracle_q8_0_blocks_from_split(const int8_t* q, const uint16_t* d, int K, int N, uint8_t* blocks) {
    const int nb = K / 32;
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < nb; ++b) {
            uint8_t* blk = blocks + ((size_t)n * nb + b) * 34;
            const uint16_t s = d[(size_t)n * nb + b];
            blk[0] = (uint8_t)(s & 0xFFu);
            blk[1] = (uint8_t)(s >> 8);
            for (int j = 0; j < 32; ++j) blk[2 + j] = (uint8_t)q[(size_t)n * K + (size_t)b * 32 + j];
        }
    }
}
