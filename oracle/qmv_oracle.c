/*
 * qmv_oracle.c -- CPU oracle for the affine group-quantized mat-vec (qmv).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's
 * CPU-baseline / reference leg may load this library. The product path
 * (the CUDA library) never calls it, links it or shares code with it.
 *
 * Plain, slow, obviously correct C. No SIMD, no blocking, no reordering
 * beyond what the definitions below state. Floating point contraction is
 * disabled at build time (-ffp-contract=off) so every operation rounds as
 * written.
 *
 * What is computed (y[m, n] for every vector m and output row n):
 *
 *   w[n, i] = s[n, g(i)] * q[n, i] + b[n, g(i)],   g(i) = i / group_size
 *   y[m, n] = sum_i w[n, i] * x[m, i]
 *
 * "Affine" quantization with one scale and one bias per group of
 * group_size consecutive weights along K: group_quantized_mat pages,
 * mlxcel issue #1289 section "Correction to the obvious sketch: qdot does
 * not dequantize" (the form scale*q + bias and its two summation orders),
 * and mlxcel PR #1681 section "Not covered" (one scale and one bias per
 * group, applied once per group).
 *
 * Field layout: bits-wide unsigned fields packed little-endian into uint32
 * words, field j of a word at bits [bits*j, bits*j + bits), so field 0 sits
 * in the low bits. Issue #1289 "Correction..." (the 4-bit masks 0x000f for
 * element 4i and 0x00f0 for element 4i+1) and llama.cpp PR #159 "How"
 * ("plain bit packing keeps field 0 in the low bits").
 *
 * Mutation hooks: building with -DORACLE_MUTANT=k plants one deliberate
 * mistake (k = 1..7, listed at each hook). The pin tests build these
 * variants on the CPU and check that some pin fails for each, which shows
 * the pins can see that kind of mistake. The default build has none.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

int oracle_mutant(void) { return ORACLE_MUTANT; }

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 is the upper 16 bits of an IEEE-754 binary32, so widening is exact. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

double oracle_bf16_to_f64(uint16_t h) { return (double)oracle_bf16_to_f32(h); }

/* binary32 -> bf16, round to nearest, ties to even, on the 16 dropped bits.
 * Infinities pass through; a NaN stays a (quiet) NaN. A carry out of the
 * significand correctly moves to the next binade or to infinity. */
uint16_t oracle_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {
        if (u & 0x007fffffu)
            return (uint16_t)((u >> 16) | 0x0040u);
        return (uint16_t)(u >> 16);
    }
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

void oracle_f32_to_bf16_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16_rne(in[i]);
}

/* ------------------------------------------------------- field layout -- */

/* Value of element i of a row stored as packed words (field 0 = low bits). */
uint32_t oracle_field(const uint32_t *row_words, int64_t i, int bits)
{
    int64_t per_word = 32 / bits;
    uint32_t word = row_words[i / per_word];
    int shift = (int)(i % per_word) * bits;
#if ORACLE_MUTANT == 1 /* mistake: fields read from the high end of the word */
    shift = (int)(per_word - 1 - i % per_word) * bits;
#endif
    return (word >> shift) & ((1u << bits) - 1u);
}

/* Pack q[N, K] (each value < 2^bits) into words[N, K*bits/32]. */
void oracle_pack(const uint8_t *q, uint32_t *words, int64_t N, int64_t K, int bits)
{
    int64_t per_word = 32 / bits;
    int64_t wpr = K / per_word;
    memset(words, 0, (size_t)(N * wpr) * sizeof(uint32_t));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t i = 0; i < K; ++i) {
            uint32_t v = (uint32_t)q[n * K + i] & ((1u << bits) - 1u);
            words[n * wpr + i / per_word] |= v << ((i % per_word) * bits);
        }
}

/* Every field of one byte, read with shifts and masks: out[j] = field j. */
void oracle_byte_fields(uint8_t byte, int bits, int32_t *out)
{
    uint32_t w = byte;
    for (int j = 0; j < 8 / bits; ++j)
        out[j] = (int32_t)oracle_field(&w, j, bits);
}

/* The same fields by the float-floor chain of llama.cpp PR #159, "How":
 * a byte b is a base-4 fraction of 256; with u = b/256 and g_k = floor(4^k u)
 * (exact in binary32) the fields come out from the top: g_1 is field 3,
 * g_2 - 4 g_1 field 2, g_3 - 4 g_2 field 1 and b - 4 g_3 field 0.
 * For 4-bit fields the base-16 analogue has one step: g_1 = floor(16 u) is
 * field 1 and b - 16 g_1 field 0. Arithmetic is binary32, as on the page. */
void oracle_byte_fields_floatfloor(uint8_t byte, int bits, int32_t *out)
{
    float b = (float)byte;
    float u = b / 256.0f;
    if (bits == 2) {
        float g1 = floorf(4.0f * u);
        float g2 = floorf(16.0f * u);
        float g3 = floorf(64.0f * u);
        out[3] = (int32_t)g1;
        out[2] = (int32_t)(g2 - 4.0f * g1);
        out[1] = (int32_t)(g3 - 4.0f * g2);
        out[0] = (int32_t)(b - 4.0f * g3);
    } else {
        float g1 = floorf(16.0f * u);
        out[1] = (int32_t)g1;
        out[0] = (int32_t)(b - 16.0f * g1);
    }
}

/* -------------------------------------------------------- qmv, fp64 -- */

static double weight_f64(const uint32_t *row_words, const uint16_t *s_row,
                         const uint16_t *b_row, int64_t i, int bits, int gs)
{
    int64_t g = i / gs;
#if ORACLE_MUTANT == 2 /* mistake: group index taken with twice the group size */
    g = i / (2 * gs);
#endif
    double s = oracle_bf16_to_f64(s_row[g]);
    double b = oracle_bf16_to_f64(b_row[g]);
#if ORACLE_MUTANT == 3 /* mistake: bias dropped */
    b = 0.0;
#endif
    return s * (double)oracle_field(row_words, i, bits) + b;
}

/* y[m, n] = sum_i (s q + b) x: dequantize, then dot (issue #1289,
 * "Correction...": the form sum_i (scale*q_i + bias)*x_i). The reference
 * form for every tolerance check. */
void oracle_qmv_f64_dequant(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                            const uint16_t *x, double *y,
                            int64_t M, int64_t N, int64_t K, int bits, int gs)
{
    int64_t wpr = K * bits / 32, G = K / gs;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i) {
                double w = weight_f64(wq + n * wpr, scales + n * G, biases + n * G, i, bits, gs);
                int64_t xi = i;
#if ORACLE_MUTANT == 4 /* mistake: activation index transposed within the group */
                xi = (i / gs) * gs + (gs - 1 - i % gs);
#endif
                acc += w * oracle_bf16_to_f64(x[m * K + xi]);
            }
            y[m * N + n] = acc;
        }
}

/* y[m, n] = sum_g ( s_g * sum_{i in g} q_i x_i + b_g * sum_{i in g} x_i ):
 * the factored form (issue #1289 "Correction...": scale*(sum q x) +
 * bias*(sum x); PR #1681 "Not covered": per group). */
void oracle_qmv_f64_factored(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                             const uint16_t *x, double *y,
                             int64_t M, int64_t N, int64_t K, int bits, int gs)
{
    int64_t wpr = K * bits / 32, G = K / gs;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                double dot = 0.0, sx = 0.0;
                for (int64_t t = 0; t < gs; ++t) {
                    int64_t i = g * gs + t;
                    double xv = oracle_bf16_to_f64(x[m * K + i]);
                    dot += (double)oracle_field(wq + n * wpr, i, bits) * xv;
                    sx += xv;
                }
                double s = oracle_bf16_to_f64(scales[n * G + g]);
                double b = oracle_bf16_to_f64(biases[n * G + g]);
#if ORACLE_MUTANT == 5 /* mistake: sign of the bias term flipped */
                b = -b;
#endif
#if ORACLE_MUTANT == 6 /* mistake: scale and bias swapped */
                { double t_ = s; s = b; b = t_; }
#endif
                acc += s * dot + b * sx;
            }
            y[m * N + n] = acc;
        }
}

/* T[m, n] = sum_i |w_i x_i| in fp64, the scale of the acceptance bound
 * |y_gpu - y| <= 8e-3 * T + 1e-5. */
void oracle_qmv_abs_terms(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                          const uint16_t *x, double *t,
                          int64_t M, int64_t N, int64_t K, int bits, int gs)
{
    int64_t wpr = K * bits / 32, G = K / gs;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i) {
                double w = weight_f64(wq + n * wpr, scales + n * G, biases + n * G, i, bits, gs);
                acc += fabs(w * oracle_bf16_to_f64(x[m * K + i]));
            }
            t[m * N + n] = acc;
        }
}

/* ------------------------------------------------ qmv, fp32 factored -- */

/* The factored form evaluated in binary32 with bf16 output: per group an
 * fp32 running dot (products q*x are exact in fp32) and running sum of x,
 * then acc += s*dot + b*sx, then round to bf16 (nearest even). Element and
 * group order is plain increasing index. This is the CPU baseline that is
 * timed beside the GPU; it is also a sanity check within tolerance. */
struct f32_job {
    const uint32_t *wq; const uint16_t *s; const uint16_t *b; const uint16_t *x;
    uint16_t *y; float *y32; int64_t M, N, K, n0, n1; int bits, gs;
};

static void *f32_worker(void *arg)
{
    struct f32_job *j = (struct f32_job *)arg;
    int64_t wpr = j->K * j->bits / 32, G = j->K / j->gs;
    for (int64_t n = j->n0; n < j->n1; ++n)
        for (int64_t m = 0; m < j->M; ++m) {
            float acc = 0.0f;
            for (int64_t g = 0; g < G; ++g) {
                float dot = 0.0f, sx = 0.0f;
                for (int64_t t = 0; t < j->gs; ++t) {
                    int64_t i = g * j->gs + t;
                    float xv = oracle_bf16_to_f32(j->x[m * j->K + i]);
                    float qv = (float)oracle_field(j->wq + n * wpr, i, j->bits);
                    dot = dot + qv * xv;
                    sx = sx + xv;
                }
                float s = oracle_bf16_to_f32(j->s[n * G + g]);
                float b = oracle_bf16_to_f32(j->b[n * G + g]);
                acc = acc + (s * dot + b * sx);
            }
            if (j->y32) j->y32[m * j->N + n] = acc;
            if (j->y) j->y[m * j->N + n] = oracle_f32_to_bf16_rne(acc);
#if ORACLE_MUTANT == 7 /* mistake: bf16 output truncated instead of rounded */
            if (j->y) { uint32_t u; memcpy(&u, &acc, 4); j->y[m * j->N + n] = (uint16_t)(u >> 16); }
#endif
        }
    return NULL;
}

/* Rows are split into nthreads contiguous blocks, one pthread each. y (bf16
 * bits) and y32 (the fp32 value before rounding) may each be NULL.
 * Returns the number of threads used. */
int oracle_qmv_f32_factored(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                            const uint16_t *x, uint16_t *y, float *y32,
                            int64_t M, int64_t N, int64_t K, int bits, int gs, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = (int)N;
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    struct f32_job *jobs = (struct f32_job *)calloc((size_t)nthreads, sizeof(struct f32_job));
    if (!tid || !jobs) { free(tid); free(jobs); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        struct f32_job j = {wq, scales, biases, x, y, y32, M, N, K,
                            N * t / nthreads, N * (t + 1) / nthreads, bits, gs};
        jobs[t] = j;
    }
    char *started = (char *)calloc((size_t)nthreads, 1);
    if (!started) { free(tid); free(jobs); return -1; }
    int used = 1;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, f32_worker, &jobs[t]) == 0) { started[t] = 1; ++used; }
        else f32_worker(&jobs[t]);
    }
    f32_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (started[t]) pthread_join(tid[t], NULL);
    free(started);
    free(tid);
    free(jobs);
    return used;
}

/* ------------------------------------------------ mxfp4 (the fp mode) -- */

/*
 * The pages name a second phase, an order-preserving streamed qmv for the
 * fp quantization modes ("mxfp4", mlxcel issue #1289, section "Scope
 * limits, stated honestly"), without giving the format. The plain reading taken here is the
 * OCP Microscaling (MX) v1.0 MXFP4 format:
 *
 *   element  E2M1, 4 bits: sign (bit 3), exponent (bits 2..1, bias 1),
 *            mantissa (bit 0); exponent field 0 is subnormal (no implicit 1).
 *   scale    E8M0, one unsigned byte per block of 32 consecutive elements
 *            along K: 2^(e - 127); e = 255 is NaN.
 *
 *   w[n, i] = scale[n, i/32] * e2m1(q[n, i])
 *   y[m, n] = sum_i w[n, i] * x[m, i]
 *
 * The 4-bit codes use the same packed layout as the affine 4-bit fields
 * (field j of a word at bits [4j, 4j+4)).
 */

double oracle_e2m1_to_f64(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
#if ORACLE_MUTANT == 8 /* mistake: sign bit ignored */
    sign = 0;
#endif
    double mag;
#if ORACLE_MUTANT == 9 /* mistake: exponent field 0 read as a normal number */
    mag = ldexp(1.0 + 0.5 * m, e - 1);
#else
    if (e == 0)
        mag = 0.5 * m; /* subnormal: (m / 2) * 2^(1 - bias) */
    else
        mag = ldexp(1.0 + 0.5 * m, e - 1); /* (1 + m / 2) * 2^(e - bias) */
#endif
    return sign ? -mag : mag;
}

double oracle_e8m0_to_f64(uint8_t e)
{
    if (e == 255)
        return NAN;
    int bias = 127;
#if ORACLE_MUTANT == 10 /* mistake: exponent bias off by one */
    bias = 128;
#endif
    return ldexp(1.0, (int)e - bias);
}

static double mx_weight_f64(const uint32_t *row_words, const uint8_t *s_row, int64_t i, int64_t B)
{
    int64_t blk = i / 32;
#if ORACLE_MUTANT == 11 /* mistake: neighbouring blocks' scales exchanged */
    if ((blk ^ 1) < B)
        blk ^= 1;
#endif
    (void)B;
    return oracle_e8m0_to_f64(s_row[blk]) * oracle_e2m1_to_f64((uint8_t)oracle_field(row_words, i, 4));
}

/* y[m, n] = sum_i (scale * e2m1(q)) x: dequantize, then dot, in fp64. */
void oracle_mxfp4_qmv_f64(const uint32_t *wq, const uint8_t *scales, const uint16_t *x, double *y,
                          int64_t M, int64_t N, int64_t K)
{
    int64_t wpr = K / 8, B = K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i)
                acc += mx_weight_f64(wq + n * wpr, scales + n * B, i, B) * oracle_bf16_to_f64(x[m * K + i]);
            y[m * N + n] = acc;
        }
}

/* T[m, n] = sum_i |w_i x_i| in fp64, the scale of the acceptance bound. */
void oracle_mxfp4_abs_terms(const uint32_t *wq, const uint8_t *scales, const uint16_t *x, double *t,
                            int64_t M, int64_t N, int64_t K)
{
    int64_t wpr = K / 8, B = K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i)
                acc += fabs(mx_weight_f64(wq + n * wpr, scales + n * B, i, B) * oracle_bf16_to_f64(x[m * K + i]));
            t[m * N + n] = acc;
        }
}
