/*
 * CPU ORACLE for the 4-bit weight-only linear layer -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously correct definition of what the GPU
 * library computes.  Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table or
 * helper with the CUDA library: every decode below is written from the format
 * definitions, one weight at a time.
 *
 * Sources (web pages; cited by title and section):
 *   [INT4]  "rumik-oss-1-int4", section "Format (rumik-int4-g128-minmax-v1)":
 *           qweight uint8 [N, K/2], two 4-bit codes per byte, the LOW nibble holds
 *           the EVEN column; scale and min fp16 [N, K/128];
 *           w[n,k] = code[n,k] * scale[n, k/128] + min[n, k/128].
 *   [NVFP4] "VoxCPM2 NVFP4 (GPTQ)", section "NVFP4 settings": 4-bit float (E2M1)
 *           weights, symmetric, group size 16, per-group scales in float8_e4m3fn,
 *           one weight_global_scale per matrix; activations stay BF16 (no
 *           input_global_scale).
 *   [HEAD]  "Rumik TTS Fast Inference", section "What Made It Faster" and its
 *           Figure 3: the output projection restricted to the current codebook,
 *           2,048 code rows plus the end token (2,049 rows).
 *
 * Readings where the pages are silent (each one is also listed in the design
 * notes of the repository):
 *   - int4 codes are unsigned 0..15 (min/max affine form); the HIGH nibble is the
 *     odd column.
 *   - A decoded weight is the exact value of the formula rounded ONCE to fp32
 *     (round-to-nearest-even).  For int4, code*scale is exact in fp32 already, so
 *     this is also fp32(code*scale) + min with one rounding.  For NVFP4 the exact
 *     product E2M1(code) * e4m3(scale) * global is rounded once to fp32; this
 *     equals fp32((code*scale) * global) because code*scale is exact.
 *   - NVFP4 packing reuses the int4 nibble order (low nibble = even column), codes
 *     [N, K/2]; e4m3 scales are row-major [N, K/16]; the global scale MULTIPLIES.
 *   - E2M1 bit layout: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa
 *     (OCP Microscaling Formats spec v1.0, FP4 E2M1).  e4m3fn: bias 7, no
 *     infinities, S.1111.111 is NaN (same spec, FP8 E4M3).
 *   - The linear layer accumulates x[m,k] * w[n,k] in fp64 and returns fp64,
 *     unrounded.
 *   - [INT8] "Rumik TTS Fast Inference", "What Made It Faster": INT8 weight-only
 *     decode projections, layout unstated.  Reading (the int8 scheme [EMB] gives
 *     for the same model family): qweight int8 [N, K], one fp16 scale per output
 *     row, w[n, k] = q[n, k] * scale[n], exact in fp32.
 *   - [EMB] "rumik-oss-1-int4", "Format": embed_tokens qweight int8 [V, 2048],
 *     scale fp16 [V].  Reading: signed two's-complement codes, one symmetric scale
 *     per row, e[t, k] = q[t, k] * scale[t] (exact in fp64); an id outside
 *     0 .. V-1 gives a row of zeros.
 *   - Quantisers (round-to-nearest, from BF16 weights; the pages' own checkpoints
 *     were made with min/max rounding [INT4] and with GPTQ [NVFP4] -- GPTQ's
 *     error feedback is out of scope, the format is the same):
 *       int4-g128: per group of 128 columns lo = min, hi = max;
 *         scale = fp16((hi - lo) / 15), min = fp16(lo), code = clamp(rint((w -
 *         min) / scale), 0, 15), code 0 when the fp16 scale is 0.
 *       NVFP4: G = amax(W) / (6 * 448) (1 when amax is 0), per group of 16
 *         columns s = e4m3((amax_g / 6) / G) (round to nearest even, saturating
 *         at 448), S = e4m3(s) * G, code = E2M1(w / S) (nearest, ties to even,
 *         saturating at 6; a code of magnitude 0 is stored as +0).
 *       Every step is one IEEE fp32 operation rounded to nearest even; the
 *       conversions to fp16, e4m3 and E2M1 are written out below from the
 *       formats' definitions.
 *
 * Build: plain C99 with OpenMP over output rows, -ffp-contract=off so that no
 * multiply-add is fused behind the reader's back.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- scalars */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double q4o_fp16_value(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE 754 binary32. */
double q4o_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* float8_e4m3fn: 1 sign, 4 exponent bits (bias 7), 3 fraction bits, no inf,
 * exponent 15 with fraction 7 is NaN. */
double q4o_e4m3_value(uint8_t s)
{
    int sign = (s >> 7) & 1;
    int e = (s >> 3) & 0xf;
    int f = s & 0x7;
    double v;
    if (e == 0)
        v = ldexp((double)f, -9);                  /* subnormal: f/8 * 2^-6 */
    else if (e == 15 && f == 7)
        v = NAN;
    else
        v = ldexp((double)(8 + f), e - 10);        /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* E2M1: 1 sign (bit 3), 2 exponent bits (bias 1), 1 fraction bit. */
double q4o_e2m1_value(uint8_t nibble)
{
    int sign = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 0x3;
    int f = nibble & 0x1;
    double v;
    if (e == 0)
        v = 0.5 * f;                               /* subnormal: f/2 * 2^0 */
    else
        v = ldexp((double)(2 + f), e - 2);         /* (1 + f/2) * 2^(e-1) */
    return sign ? -v : v;
}

/* ------------------------------------------------------------- encoders */

/* Round-to-nearest-even of a finite double that is an exact multiple of the
 * target spacing times an integer plus a fraction: rint() under the default
 * rounding mode. */
static double rne(double v) { return nearbyint(v); }

/* fp32 -> IEEE binary16, round to nearest even, overflow to infinity. */
uint16_t q4o_f32_to_fp16(float x)
{
    if (isnan(x))
        return 0x7e00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (a >= 65520.0)                               /* half-way above 65504 and beyond */
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {                      /* subnormal: multiples of 2^-24 */
        double m = rne(a * ldexp(1.0, 24));         /* 0 .. 1024 (1024 = smallest normal) */
        return sign | (uint16_t)m;
    }
    int e;
    frexp(a, &e);                                   /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                         /* 2^e <= a < 2^(e+1) */
    double m = rne(a * ldexp(1.0, 10 - e));         /* 1024 .. 2048 */
    if (m == 2048.0) {
        m = 1024.0;
        e += 1;
    }
    if (e + 15 >= 31)
        return sign | 0x7c00;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)m - 1024));
}

/* fp32 -> float8_e4m3fn, round to nearest even, saturating at +-448; NaN -> 0x7f. */
uint8_t q4o_f32_to_e4m3(float x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a < ldexp(1.0, -6)) {                       /* subnormal: multiples of 2^-9 */
        double m = rne(a * ldexp(1.0, 9));          /* 0 .. 8 (8 = smallest normal) */
        return sign | (uint8_t)m;
    }
    if (a >= 448.0)
        return sign | 0x7e;
    int e;
    frexp(a, &e);
    e -= 1;
    double m = rne(a * ldexp(1.0, 3 - e));          /* 8 .. 16 */
    if (m == 16.0) {
        m = 8.0;
        e += 1;
    }
    /* a < 448 = 1.75 * 2^8, so e <= 8 and, for e == 8, m <= 14 */
    return sign | (uint8_t)(((e + 7) << 3) | ((int)m - 8));
}

/* fp32 -> E2M1 nibble (bit 3 sign), nearest with ties to even, saturating at
 * +-6; a result of magnitude 0 is returned as +0 (code 0). */
uint8_t q4o_f32_to_e2m1(float x)
{
    double a = fabs((double)x);
    uint8_t mag;
    if (a < 1.0) {                                  /* subnormal: multiples of 0.5 */
        mag = (uint8_t)rne(a * 2.0);                /* 0, 1, 2 (2 = 1.0) */
    } else if (a >= 6.0) {
        mag = 7;
    } else {
        int e;
        frexp(a, &e);
        e -= 1;                                     /* 0 .. 2 */
        double m = rne(a * ldexp(1.0, 1 - e));      /* 2 .. 4 */
        if (m == 4.0) {
            m = 2.0;
            e += 1;
        }
        mag = (e > 2) ? 7 : (uint8_t)(((e + 1) << 1) | ((int)m - 2));
    }
    if (mag == 0)
        return 0;
    return (signbit(x) ? 8 : 0) | mag;
}

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* The 4-bit code of column k in a row of packed bytes: the low nibble holds the
 * even column, the high nibble the odd column [INT4]. */
static unsigned code_at(const uint8_t *row_bytes, int64_t k)
{
    uint8_t byte = row_bytes[k / 2];
    return (k % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
}

/* ------------------------------------------------------------- dequantise */

/* One int4-g128 weight: code * scale + min, exact, rounded once to fp32 [INT4]. */
static float int4_weight(const uint8_t *qweight, const uint16_t *scale,
                         const uint16_t *minv, int64_t K, int64_t n, int64_t k)
{
    int64_t groups = K / 128;
    unsigned c = code_at(qweight + n * (K / 2), k);
    double s = q4o_fp16_value(scale[n * groups + k / 128]);
    double m = q4o_fp16_value(minv[n * groups + k / 128]);
    return (float)((double)c * s + m);
}

/* One NVFP4 weight: E2M1(code) * e4m3(group scale) * global, exact, rounded once
 * to fp32 [NVFP4]. */
static float nvfp4_weight(const uint8_t *codes, const uint8_t *scale_e4m3,
                          float global_scale, int64_t K, int64_t n, int64_t k)
{
    int64_t groups = K / 16;
    double c = q4o_e2m1_value((uint8_t)code_at(codes + n * (K / 2), k));
    double s = q4o_e4m3_value(scale_e4m3[n * groups + k / 16]);
    return (float)(c * s * (double)global_scale);
}

void q4o_dequant_int4g128(const uint8_t *qweight, const uint16_t *scale,
                          const uint16_t *minv, int64_t N, int64_t K, float *w)
{
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = int4_weight(qweight, scale, minv, K, n, k);
}

void q4o_dequant_nvfp4(const uint8_t *codes, const uint8_t *scale_e4m3,
                       float global_scale, int64_t N, int64_t K, float *w)
{
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = nvfp4_weight(codes, scale_e4m3, global_scale, K, n, k);
}

/* ------------------------------------------------------------------ linear */

/* y[m,n] = sum_k x[m,k] * w[n,k] in fp64, x bf16 [M,K] row-major.  Also returns
 * sum_k |x[m,k] * w[n,k]| (the scale of the per-element tolerance) when absy is
 * not NULL.  Each row of weights is decoded into a scratch row first. */
/* One INT8 weight: q * scale, exact in fp32 [INT8]. */
static float int8_weight(const uint8_t *qweight, const uint16_t *scale, int64_t K, int64_t n,
                         int64_t k)
{
    return (float)((double)(int8_t)qweight[n * K + k] * q4o_fp16_value(scale[n]));
}

void q4o_dequant_int8(const int8_t *qweight, const uint16_t *scale, int64_t N, int64_t K,
                      float *w)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = int8_weight((const uint8_t *)qweight, scale, K, n, k);
}

static void linear_rows(int layout, const uint16_t *x, const uint8_t *packed,
                        const void *scale, const uint16_t *minv, float global_scale,
                        int64_t M, int64_t N, int64_t K, double *y, double *absy)
{
    #pragma omp parallel
    {
        float *wrow = (float *)malloc((size_t)K * sizeof(float));
        #pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t k = 0; k < K; ++k)
                wrow[k] = (layout == 0)
                    ? int4_weight(packed, (const uint16_t *)scale, minv, K, n, k)
                    : (layout == 1)
                    ? nvfp4_weight(packed, (const uint8_t *)scale, global_scale, K, n, k)
                    : int8_weight(packed, (const uint16_t *)scale, K, n, k);
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0, aacc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double p = q4o_bf16_value(x[m * K + k]) * (double)wrow[k];
                    acc += p;
                    aacc += fabs(p);
                }
                y[m * N + n] = acc;
                if (absy)
                    absy[m * N + n] = aacc;
            }
        }
        free(wrow);
    }
}

void q4o_linear_int8(const uint16_t *x_bf16, const int8_t *qweight, const uint16_t *scale_f16,
                     int64_t M, int64_t N, int64_t K, double *y, double *absy)
{
    linear_rows(2, x_bf16, (const uint8_t *)qweight, scale_f16, NULL, 0.0f, M, N, K, y, absy);
}

void q4o_linear_int4g128(const uint16_t *x_bf16, const uint8_t *qweight,
                         const uint16_t *scale_f16, const uint16_t *min_f16,
                         int64_t M, int64_t N, int64_t K, double *y, double *absy)
{
    linear_rows(0, x_bf16, qweight, scale_f16, min_f16, 0.0f, M, N, K, y, absy);
}

void q4o_linear_nvfp4(const uint16_t *x_bf16, const uint8_t *codes,
                      const uint8_t *scale_e4m3, float global_scale,
                      int64_t M, int64_t N, int64_t K, double *y, double *absy)
{
    linear_rows(1, x_bf16, codes, scale_e4m3, NULL, global_scale, M, N, K, y, absy);
}

/* ---------------------------------------------------------- restricted head */

/* logits[m,j] = sum_k h[m,k] * head[r_j,k] in fp64, where r_j = row_begin + j for
 * j < n_rows and r_{n_rows} = extra_row when extra_row >= 0 [HEAD].  head is bf16
 * [R_total, H] row-major; logits has n_rows + (extra_row >= 0) columns. */
void q4o_head_restricted(const uint16_t *h_bf16, const uint16_t *head_bf16,
                         int64_t row_begin, int64_t n_rows, int64_t extra_row,
                         int64_t M, int64_t H, double *logits, double *abslog)
{
    int64_t cols = n_rows + (extra_row >= 0 ? 1 : 0);
    #pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < cols; ++j) {
        int64_t r = (j < n_rows) ? row_begin + j : extra_row;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < H; ++k) {
                double p = q4o_bf16_value(h_bf16[m * H + k]) *
                           q4o_bf16_value(head_bf16[r * H + k]);
                acc += p;
                aacc += fabs(p);
            }
            logits[m * cols + j] = acc;
            if (abslog)
                abslog[m * cols + j] = aacc;
        }
    }
}

/* Array forms of the three encoders (for the tests). */
void q4o_f32_to_fp16_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = q4o_f32_to_fp16(x[i]);
}
void q4o_f32_to_e4m3_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = q4o_f32_to_e4m3(x[i]);
}
void q4o_f32_to_e2m1_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = q4o_f32_to_e2m1(x[i]);
}

/* -------------------------------------------------------------- quantise */

/* int4-g128 min/max round-to-nearest quantiser [INT4]: w_bf16 [N, K] ->
 * qweight [N, K/2] (low nibble = even column), scale and min fp16 [N, K/128]. */
void q4o_quantize_int4g128(const uint16_t *w_bf16, int64_t N, int64_t K, uint8_t *qweight,
                           uint16_t *scale, uint16_t *minv)
{
    const int64_t groups = K / 128;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < groups; ++g) {
            const uint16_t *w = w_bf16 + n * K + g * 128;
            float lo = bf16_to_f32(w[0]), hi = lo;
            for (int k = 1; k < 128; ++k) {
                float v = bf16_to_f32(w[k]);
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            float range = hi - lo;                  /* one fp32 rounding */
            uint16_t s16 = q4o_f32_to_fp16(range / 15.0f);
            uint16_t m16 = q4o_f32_to_fp16(lo);
            scale[n * groups + g] = s16;
            minv[n * groups + g] = m16;
            float s = (float)q4o_fp16_value(s16);
            float m = (float)q4o_fp16_value(m16);
            uint8_t *row = qweight + n * (K / 2) + g * 64;
            for (int k = 0; k < 128; ++k) {
                int c = 0;
                if (s > 0.0f) {
                    float d = bf16_to_f32(w[k]) - m;  /* fp32 */
                    float q = d / s;                  /* fp32 */
                    double r = rne((double)q);
                    c = r < 0.0 ? 0 : (r > 15.0 ? 15 : (int)r);
                }
                if (k % 2 == 0)
                    row[k / 2] = (uint8_t)c;
                else
                    row[k / 2] |= (uint8_t)(c << 4);
            }
        }
    }
}

/* NVFP4 round-to-nearest quantiser [NVFP4]: w_bf16 [N, K] -> E2M1 codes [N, K/2]
 * (low nibble = even column), e4m3 group scales [N, K/16], fp32 global scale. */
void q4o_quantize_nvfp4(const uint16_t *w_bf16, int64_t N, int64_t K, uint8_t *codes,
                        uint8_t *scale_e4m3, float *global_scale)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < N * K; ++i) {
        float a = fabsf(bf16_to_f32(w_bf16[i]));
        if (a > amax) amax = a;
    }
    const float G = amax > 0.0f ? amax / 2688.0f : 1.0f;   /* 2688 = 6 * 448 */
    *global_scale = G;
    const int64_t groups = K / 16;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < groups; ++g) {
            const uint16_t *w = w_bf16 + n * K + g * 16;
            float ag = 0.0f;
            for (int k = 0; k < 16; ++k) {
                float a = fabsf(bf16_to_f32(w[k]));
                if (a > ag) ag = a;
            }
            float t = ag / 6.0f;
            uint8_t s8 = q4o_f32_to_e4m3(t / G);
            scale_e4m3[n * groups + g] = s8;
            float S = (float)q4o_e4m3_value(s8) * G;          /* fp32 product */
            uint8_t *row = codes + n * (K / 2) + g * 8;
            for (int k = 0; k < 16; ++k) {
                uint8_t c = 0;
                if (S > 0.0f)
                    c = q4o_f32_to_e2m1(bf16_to_f32(w[k]) / S);
                if (k % 2 == 0)
                    row[k / 2] = c;
                else
                    row[k / 2] |= (uint8_t)(c << 4);
            }
        }
    }
}

/* ------------------------------------------------------------- embedding */

/* Gather and dequantise embedding rows [EMB]: out[m, k] = q[ids[m], k] *
 * scale[ids[m]] in fp64 (exact), zeros for an id outside 0 .. V-1. */
void q4o_embedding_int8(const int32_t *ids, const int8_t *qweight, const uint16_t *scale,
                        int64_t M, int64_t V, int64_t H, double *out)
{
    for (int64_t m = 0; m < M; ++m) {
        const int64_t t = ids[m];
        for (int64_t k = 0; k < H; ++k) {
            if (t < 0 || t >= V)
                out[m * H + k] = 0.0;
            else
                out[m * H + k] = (double)qweight[t * H + k] * q4o_fp16_value(scale[t]);
        }
    }
}

int q4o_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
