/*
 * qmm_oracle.c -- the CPU oracle for the weight-only quantized matrix product.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline do.  It shares no header, helper, table or constant with the CUDA
 * library under quantized_weight_gb300/csrc/.
 *
 * It is deliberately plain and slow: every output is a double-precision sum,
 * in k order, of exactly dequantized weights times the activations, following
 * the fused "dequantize one block, then accumulate it" loop of
 *   "I Built an LLM Inference Engine on a 15 year old GPU ..." (medium.rebeauty-writing.com),
 *   section "Optimization 4: Quantized Kernels" (the per-block dequantize-then-dot loop),
 * with the affine formula  dequantized = q * scale + min  of the same page's
 * section "Quantization: The Model Doesn't Run on INT4".
 *
 * Formats (the pages leave bit order and layout open; the reading used is):
 *   W is [N, K] row-major, output feature n has the K inputs of row n.
 *   Codes are packed little-endian into 32-bit words: element k of a row is in
 *   word k / (32/bits) of that row, at bit offset bits * (k mod (32/bits)).
 *     bits = 4 : affine, w = s*q + b, q in 0..15   (group-64 affine INT4 codes,
 *                "Pushing the limits of legacy hardware", first section)
 *     bits = 8 : symmetric, w = s*q, q a two's-complement int8
 *                ("... Tesla C2075 ..." paper, section 2.3 Quantization and residency)
 *     bits = 1 : sign, w = s*(2b - 1): bit 1 is +1, bit 0 is -1
 *                ("A 27B model on two 4GB Maxwell GPUs", binary Q1 weights with FP16 scales)
 *   Scales and biases are IEEE binary16 bit patterns, [N, K/group] row-major;
 *   group g of row n covers k in [g*group, (g+1)*group).
 *   y[m, n] = sum_k x[m, k] * w[n, k]  (y = x * dequant(W)^T).
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 * Compile with -O2 -ffp-contract=off and no fast-math, so that every double
 * operation written here is one IEEE operation.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);     /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 128), e - 134);     /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* ------------------------------------------------------------ encoders */

/* float32 -> IEEE 754 binary16, round to nearest, ties to even; overflow to
 * infinity, gradual underflow to subnormals, NaN to a quiet NaN with the
 * sign kept (0x7E00 | sign).  Written from the two formats' bit layouts. */
uint16_t oracle_float_to_half(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    int e = (int)((u >> 23) & 0xFF);
    uint32_t m = u & 0x7FFFFFu;
    if (e == 255) return (uint16_t)(sign | (m ? 0x7E00u : 0x7C00u));
    if (e == 0 && m == 0) return sign;
    /* value = sig * 2^(exp2) with sig an integer of up to 24 bits */
    uint32_t sig = (e == 0) ? m : (m | 0x800000u);
    int exp2 = (e == 0) ? -149 : e - 150;
    /* target: binary16 value = hsig * 2^hexp, hexp >= -24 (subnormal step),
     * normal numbers keep 11 significant bits */
    int msb = 31;
    while (!((sig >> msb) & 1u)) msb--;             /* position of the leading bit */
    int top = exp2 + msb;                           /* value in [2^top, 2^(top+1)) */
    int hexp = top - 10;                            /* ulp exponent for 11 bits */
    if (hexp < -24) hexp = -24;                     /* subnormal range */
    int shift = hexp - exp2;                        /* bits of sig to drop */
    uint32_t q;
    if (shift <= 0) {
        q = sig << (-shift);                        /* exact */
    } else if (shift > 31) {
        q = 0;                                      /* far below half the smallest subnormal */
    } else {
        uint32_t rem = sig & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        q = sig >> shift;
        if (rem > half || (rem == half && (q & 1u))) q++;
    }
    /* q * 2^hexp; q may have carried to 2^11 (or reached 2^10 from a subnormal) */
    if (q == 0) return sign;
    int E = hexp + 25;                              /* biased exponent if q in [2^10, 2^11) */
    if (q >= 2048u) { q >>= 1; E++; }               /* carry: q was exactly 2^11 */
    if (q < 1024u) return (uint16_t)(sign | q);     /* subnormal (hexp == -24) */
    if (E >= 31) return (uint16_t)(sign | 0x7C00u); /* overflow */
    return (uint16_t)(sign | ((uint32_t)E << 10) | (q & 0x3FFu));
}

/* ------------------------------------------------------------ packing */

static int bits_ok(int bits) { return bits == 1 || bits == 4 || bits == 8; }

static int64_t words_per_row(int64_t K, int bits) { return K * bits / 32; }

/* codes: [N, K], one code per byte (0..15 for bits=4; the int8 bit pattern
 * for bits=8; 0 or 1 for bits=1).  packed: [N, K*bits/32] 32-bit words. */
int oracle_pack(const uint8_t *codes, uint32_t *packed, int64_t N, int64_t K, int bits)
{
    if (!bits_ok(bits) || N < 0 || K < 0 || K % 32 != 0) return -1;
    int64_t per_word = 32 / bits;
    uint32_t mask = (1u << bits) - 1u;
    int64_t wpr = words_per_row(K, bits);
    for (int64_t n = 0; n < N; n++) {
        for (int64_t w = 0; w < wpr; w++) {
            uint32_t word = 0;
            for (int64_t j = 0; j < per_word; j++) {
                uint32_t c = codes[n * K + w * per_word + j];
                if ((c & mask) != c) return -2;    /* code does not fit in `bits` */
                word |= c << (bits * j);
            }
            packed[n * wpr + w] = word;
        }
    }
    return 0;
}

/* The code of element (n, k) as an integer: 0..15, -128..127 or 0/1. */
static int code_at(const uint32_t *packed, int64_t n, int64_t k, int64_t K, int bits)
{
    int64_t per_word = 32 / bits;
    uint32_t word = packed[n * words_per_row(K, bits) + k / per_word];
    int shift = (int)(bits * (k % per_word));
    int u = (int)((word >> shift) & ((1u << bits) - 1u));
    if (bits == 8 && u >= 128) u -= 256;           /* two's complement byte */
    return u;
}

int oracle_unpack(const uint32_t *packed, uint8_t *codes, int64_t N, int64_t K, int bits)
{
    if (!bits_ok(bits) || N < 0 || K < 0 || K % 32 != 0) return -1;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++)
            codes[n * K + k] = (uint8_t)(code_at(packed, n, k, K, bits) & 0xFF);
    return 0;
}

/* ------------------------------------------------------------ dequant */

static int shape_ok(int64_t N, int64_t K, int bits, int group)
{
    if (!bits_ok(bits) || N < 0 || K < 0 || K % 32 != 0) return 0;
    if (group <= 0 || K % group != 0) return 0;
    return 1;
}

/* One weight, exactly, in double: s*q (+ b).  Exact because s*q has at most
 * 11 + 8 significant bits and s*q + b spans fewer than 53 bits. */
static double weight_at(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                        int64_t n, int64_t k, int64_t K, int bits, int group)
{
    int64_t groups = K / group;
    int64_t g = k / group;
    double s = oracle_half_to_double(scales[n * groups + g]);
    int q = code_at(packed, n, k, K, bits);
    if (bits == 4) {
        double b = oracle_half_to_double(biases[n * groups + g]);
        return s * (double)q + b;
    }
    if (bits == 8) return s * (double)q;
    return s * (double)(2 * q - 1);
}

int oracle_dequant(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                   double *w, int64_t N, int64_t K, int bits, int group)
{
    if (!shape_ok(N, K, bits, group)) return -1;
    if (bits == 4 && biases == NULL) return -1;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++)
            w[n * K + k] = weight_at(packed, scales, biases, n, k, K, bits, group);
    return 0;
}

/* ------------------------------------------------------------ the product */

/* Row n of W decoded into wrow[0..K). */
static void decode_row(double *wrow, const uint32_t *packed, const uint16_t *scales,
                       const uint16_t *biases, int64_t n, int64_t K, int bits, int group)
{
    for (int64_t k = 0; k < K; k++)
        wrow[k] = weight_at(packed, scales, biases, n, k, K, bits, group);
}

/* One output: acc = sum over groups g, over k in the group, of w[n,k]*x[m,k],
 * in double, in increasing k (wrow: row n of W, decoded). */
static double dot_row(const double *wrow, const double *xrow, int64_t K, int group)
{
    double acc = 0.0;
    for (int64_t g0 = 0; g0 < K; g0 += group)
        for (int64_t k = g0; k < g0 + group; k++)
            acc += wrow[k] * xrow[k];
    return acc;
}

typedef struct {
    const double *x;            /* [M, K] activations, already decoded to double */
    const uint32_t *packed;
    const uint16_t *scales, *biases;
    double *y;                  /* [M, N] */
    int64_t M, N, K;
    int bits, group;
    int64_t n_begin, n_end;
    double *wrow;               /* [K] this thread's decoded row */
} qmm_job;

/* Row n is decoded once and used for every token m (each weight is the
 * same value for every token, so this changes no result). */
static void *qmm_worker(void *arg)
{
    qmm_job *j = (qmm_job *)arg;
    for (int64_t n = j->n_begin; n < j->n_end; n++) {
        decode_row(j->wrow, j->packed, j->scales, j->biases, n, j->K, j->bits, j->group);
        for (int64_t m = 0; m < j->M; m++)
            j->y[m * j->N + n] = dot_row(j->wrow, j->x + m * j->K, j->K, j->group);
    }
    return NULL;
}

/* Rows n are split over `nthreads` POSIX threads; each output is computed by
 * one thread in the order above, so the result does not depend on nthreads. */
static int qmm_double_x(const double *x, const uint32_t *packed, const uint16_t *scales,
                        const uint16_t *biases, double *y, int64_t M, int64_t N, int64_t K,
                        int bits, int group, int nthreads)
{
    if (!shape_ok(N, K, bits, group) || M < 0) return -1;
    if (bits == 4 && biases == NULL) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > N) nthreads = (int)(N > 0 ? N : 1);
    pthread_t tid[256];
    qmm_job jobs[256];
    double *rows = (double *)malloc(sizeof(double) * (size_t)nthreads * (size_t)(K > 0 ? K : 1));
    if (!rows) return -3;
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (qmm_job){x, packed, scales, biases, y, M, N, K, bits, group,
                            N * t / nthreads, N * (t + 1) / nthreads, rows + (size_t)t * (size_t)(K > 0 ? K : 1)};
    }
    int started = 0;
    for (int t = 1; t < nthreads; t++) {
        if (pthread_create(&tid[t], NULL, qmm_worker, &jobs[t]) != 0) break;
        started = t;
    }
    qmm_worker(&jobs[0]);
    for (int t = 1; t <= started; t++) pthread_join(tid[t], NULL);
    for (int t = started + 1; t < nthreads; t++) qmm_worker(&jobs[t]);  /* threads that failed to start */
    free(rows);
    return 0;
}

/* x given as IEEE binary32 values (the decode GEMV's activations). */
int oracle_qmm_f32x(const float *x, const uint32_t *packed, const uint16_t *scales,
                    const uint16_t *biases, double *y, int64_t M, int64_t N, int64_t K,
                    int bits, int group, int nthreads)
{
    if (M < 0 || K < 0) return -1;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!xd) return -3;
    for (int64_t i = 0; i < M * K; i++) xd[i] = (double)x[i];
    int r = qmm_double_x(xd, packed, scales, biases, y, M, N, K, bits, group, nthreads);
    free(xd);
    return r;
}

/* x given as bfloat16 bit patterns (the prefill contraction's activations). */
int oracle_qmm_bf16x(const uint16_t *x, const uint32_t *packed, const uint16_t *scales,
                     const uint16_t *biases, double *y, int64_t M, int64_t N, int64_t K,
                     int bits, int group, int nthreads)
{
    if (M < 0 || K < 0) return -1;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!xd) return -3;
    for (int64_t i = 0; i < M * K; i++) xd[i] = oracle_bf16_to_double(x[i]);
    int r = qmm_double_x(xd, packed, scales, biases, y, M, N, K, bits, group, nthreads);
    free(xd);
    return r;
}

/* Selected outputs only: out[i] = y[ms[i], ns[i]].  For shapes whose full
 * product is too slow on a CPU; x_is_bf16 selects the activation encoding
 * (x points at float values when 0, at bfloat16 bit patterns when 1). */
int oracle_qmm_sampled(const void *x, int x_is_bf16, const uint32_t *packed,
                       const uint16_t *scales, const uint16_t *biases, const int64_t *ms,
                       const int64_t *ns, int64_t count, double *out, int64_t M, int64_t N,
                       int64_t K, int bits, int group)
{
    if (!shape_ok(N, K, bits, group) || M < 0 || count < 0) return -1;
    if (bits == 4 && biases == NULL) return -1;
    double *xrow = (double *)malloc(sizeof(double) * 2 * (size_t)(K > 0 ? K : 1));
    if (!xrow) return -3;
    double *wrow = xrow + (K > 0 ? K : 1);
    for (int64_t i = 0; i < count; i++) {
        int64_t m = ms[i], n = ns[i];
        if (m < 0 || m >= M || n < 0 || n >= N) { free(xrow); return -2; }
        for (int64_t k = 0; k < K; k++)
            xrow[k] = x_is_bf16 ? oracle_bf16_to_double(((const uint16_t *)x)[m * K + k])
                                : (double)((const float *)x)[m * K + k];
        decode_row(wrow, packed, scales, biases, n, K, bits, group);
        out[i] = dot_row(wrow, xrow, K, group);
    }
    free(xrow);
    return 0;
}

/* ------------------------------------------------------------ quantizer */

/* Affine 4-bit quantization of one block, as the quantization section of the
 * "15 year old GPU" page describes it: the block's min and max define the
 * range, scale = (max - min) / 15, every weight becomes
 * q = round((w - min) / scale) in 0..15 (rounded to nearest, halves away from
 * zero, then clamped), and  dequantized = q * scale + min.  A block whose
 * values are all equal gets scale 0 and codes 0.  All in double. */
int oracle_quantize_affine4(const double *w, int64_t count, uint8_t *q, double *scale,
                            double *minv)
{
    if (count <= 0) return -1;
    double lo = w[0], hi = w[0];
    for (int64_t i = 1; i < count; i++) {
        if (w[i] < lo) lo = w[i];
        if (w[i] > hi) hi = w[i];
    }
    double s = (hi - lo) / 15.0;
    for (int64_t i = 0; i < count; i++) {
        double r = (s > 0.0) ? round((w[i] - lo) / s) : 0.0;
        if (r < 0.0) r = 0.0;
        if (r > 15.0) r = 15.0;
        q[i] = (uint8_t)r;
    }
    *scale = s;
    *minv = lo;
    return 0;
}

/* The quantizer as the library stores its output: INT4 affine codes with
 * binary16 scale and bias per group of `group` consecutive k of a row.
 * Per group, in float32 (every operation one IEEE float operation):
 *   lo, hi  = min and max of the group's values (NaN values are skipped)
 *   scale   = binary16(RNE((hi - lo) / 15)),  bias = binary16(RNE(lo))
 *             (-0 orders below +0 in the min and max; a NaN scale or bias is
 *             stored as 0x7E00)
 *   q       = clamp(roundf((w - bias) / scale), 0, 15), halves away from zero,
 *             taken with the stored (binary16) scale and bias, so that
 *             q * scale + bias is the nearest level of the stored grid;
 *             q = 0 when the stored scale is not positive and finite, or w is NaN.
 * The float32 steps are the reading of the page's "round((w - min) / scale)"
 * for a format that stores binary16 coefficients; the decision that picks the
 * integer q is made in the same precision on the CPU and on the GPU. */
int oracle_quantize_affine4_f32(const float *w, int64_t N, int64_t K, int group, uint8_t *codes,
                                uint16_t *scales, uint16_t *biases)
{
    if (N < 0 || K < 0 || group <= 0 || K % group != 0) return -1;
    int64_t G = K / group;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t g = 0; g < G; g++) {
            const float *v = w + n * K + g * group;
            float lo = NAN, hi = NAN;
            for (int i = 0; i < group; i++) {
                float x = v[i];
                if (isnan(x)) continue;
                /* -0 counts as below +0, so the result does not depend on order */
                if (isnan(lo) || x < lo || (x == lo && signbit(x) && !signbit(lo))) lo = x;
                if (isnan(hi) || x > hi || (x == hi && !signbit(x) && signbit(hi))) hi = x;
            }
            volatile float range = hi - lo;
            volatile float s32 = range / 15.0f;
            uint16_t sh = isnan(s32) ? 0x7E00u : oracle_float_to_half(s32);
            uint16_t bh = isnan(lo) ? 0x7E00u : oracle_float_to_half(lo);
            float s = (float)oracle_half_to_double(sh), b = (float)oracle_half_to_double(bh);
            scales[n * G + g] = sh;
            biases[n * G + g] = bh;
            for (int i = 0; i < group; i++) {
                uint8_t c = 0;
                if (s > 0.0f && isfinite(s) && !isnan(v[i])) {
                    volatile float d = v[i] - b;
                    volatile float t = d / s;
                    float r = roundf(t);
                    if (isnan(r)) r = 0.0f;
                    if (r < 0.0f) r = 0.0f;
                    if (r > 15.0f) r = 15.0f;
                    c = (uint8_t)r;
                }
                codes[n * K + g * group + i] = c;
            }
        }
    }
    return 0;
}
