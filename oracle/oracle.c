/*
 * CPU oracle for the int8 quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  The CUDA product
 * path never links, calls or reads it, and this file shares no code,
 * header, table or helper with the CUDA sources.
 *
 * Every function is the plain definition written out as loops, in the
 * precision the pages fix (fp32 for scales, exact integers for codes and
 * accumulators) or in fp64 where they fix none.  Build flags:
 * -O2 -ffp-contract=off -fno-fast-math, so that no multiply-add is fused
 * and no denormal is flushed.  With OpenMP the outer loop over output rows
 * is shared among threads; every output is still computed by one thread in
 * the same order, so results do not depend on the thread count.
 *
 * Sources, cited by page title and section:
 *  [Q]  "Day 6 -- Quantize It Yourself", The mechanism, block 1: a stored
 *       tensor is q = clamp(round(w / s)) with s = absmax(group) / qmax, and
 *       reconstructs as w ~ s * q; the group can be one output channel.
 *  [RTN] same page, block 4: round-to-nearest, each weight independently.
 *  [P1] "Phase 5a: int8 weight-only quantization", Summary: per-output-
 *       channel int8 weights; the scale arithmetic is float32, not the
 *       weight's bf16/fp16 dtype; only the all-zero channel is guarded,
 *       with no dtype-dependent floor on small channels.
 *  [W8A8] "feat(quantization): support compressed-tensors W8A8 and mixed
 *       modules", Design and Supported Execution Scheme: static symmetric
 *       int8 per-channel weights, dynamic symmetric int8 per-token
 *       activations, no output-activation quantization; Summary: weight
 *       scales are loaded as FP32.
 *  [W8A16] "Day 6", block 5: weight-only int8 is dequantized inside the
 *       kernel and multiplied on bf16 math (dequantize-then-matmul).
 *  [MOE] "Phase 5a", Summary: a grouped GEMM over MoE experts with stacked
 *       [E, N, K] expert weights.
 *
 * Readings where the pages are silent: round() ties go to even; w / s is
 * one IEEE fp32 division per element; an all-zero row stores s = 1 and
 * all-zero codes; codes are clamped to the symmetric range [-127, 127]; the
 * W8A8 epilogue is ((float)acc * sx[m]) * sw[n], then + (float)bias[n],
 * rounded to bf16 once with round-to-nearest-even; the W8A16 reference keeps
 * s * q unrounded and accumulates in fp64.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_NONFINITE 1
#define ORACLE_ERR_ARG 2
#define ORACLE_ERR_OVERFLOW 3
#define ORACLE_ERR_OFFSETS 4

/* Threads of the row loops (all cores by default); returns the count in
 * effect, 1 in a build without OpenMP. */
int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static float widen_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even. */
static uint16_t narrow_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* Round to the nearest integer, ties to even, written out so that it does
 * not depend on the floating-point environment.  |t| < 2^23 here. */
static float round_half_even(float t) {
    float fl = floorf(t);
    float frac = t - fl; /* exact for |t| < 2^23 */
    if (frac > 0.5f) return fl + 1.0f;
    if (frac < 0.5f) return fl;
    return (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
}

/*
 * Per-row symmetric int8 quantization [Q][RTN][P1]: weights (one row per
 * output channel, [P1]) and activations (one row per token, [W8A8]) use the
 * same arithmetic on a different row.
 *   a    = max_k |v[r,k]|                       (fp32, exact)
 *   s[r] = a / 127  in fp32; s[r] = 1 if a == 0 (zero-channel guard)
 *   q    = clamp(round_half_even(v / s[r]), -127, 127)
 */
int oracle_quant_rows(const uint16_t* src, int64_t rows, int64_t k,
                      int8_t* q, float* s) {
    if (rows < 0 || k < 0) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < rows * k; ++i)
        if (!isfinite(widen_bf16(src[i]))) return ORACLE_ERR_NONFINITE;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* row = src + r * k;
        float a = 0.0f;
        for (int64_t j = 0; j < k; ++j) {
            float av = fabsf(widen_bf16(row[j]));
            if (av > a) a = av;
        }
        float scale = (a == 0.0f) ? 1.0f : a / 127.0f;
        s[r] = scale;
        for (int64_t j = 0; j < k; ++j) {
            float t = widen_bf16(row[j]) / scale;
            float c = round_half_even(t);
            if (c > 127.0f) c = 127.0f;
            if (c < -127.0f) c = -127.0f;
            q[r * k + j] = (int8_t)c;
        }
    }
    return ORACLE_OK;
}

/* Exact integer product acc[m,n] = sum_k qx[m,k] * qw[n,k], in int64. */
int oracle_int_acc(const int8_t* qx, const int8_t* qw, int64_t m_rows,
                   int64_t n_rows, int64_t k, int64_t* acc) {
    if (m_rows < 0 || n_rows < 0 || k < 0) return ORACLE_ERR_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < m_rows; ++m)
        for (int64_t n = 0; n < n_rows; ++n) {
            int64_t sum = 0;
            for (int64_t j = 0; j < k; ++j)
                sum += (int64_t)qx[m * k + j] * (int64_t)qw[n * k + j];
            acc[m * n_rows + n] = sum;
        }
    return ORACLE_OK;
}

/* One W8A8 output from its exact accumulator [W8A8]:
 *   f = ((float)acc * sx) * sw   (+ (float)bias),   y = bf16_rne(f). */
static int w8a8_point(int64_t acc, float sx, float sw, const uint16_t* bias,
                      int64_t n, float* f_out, uint16_t* y_out) {
    if (acc > INT32_MAX || acc < INT32_MIN) return ORACLE_ERR_OVERFLOW;
    float f = (float)(int32_t)acc;
    f = f * sx;
    f = f * sw;
    if (bias) f = f + widen_bf16(bias[n]);
    *f_out = f;
    *y_out = narrow_bf16_rne(f);
    return ORACLE_OK;
}

/* Full W8A8 epilogue over an [M, N] accumulator. */
int oracle_w8a8_epilogue(const int64_t* acc, const float* sx, const float* sw,
                         const uint16_t* bias, int64_t m_rows, int64_t n_rows,
                         float* f, uint16_t* y) {
    int err = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < m_rows; ++m)
        for (int64_t n = 0; n < n_rows; ++n) {
            int64_t i = m * n_rows + n;
            int rc = w8a8_point(acc[i], sx[m], sw[n], bias, n, &f[i], &y[i]);
            if (rc) {
#pragma omp atomic write
                err = rc;
            }
        }
    return err;
}

/* W8A8 at chosen output points (m = pm[i], n = pn[i]) of a large layer:
 * the exact accumulator and the epilogue, one dot product per point. */
int oracle_w8a8_points(const int8_t* qx, const float* sx, const int8_t* qw,
                       const float* sw, const uint16_t* bias, int64_t m_rows,
                       int64_t n_rows, int64_t k, int64_t npts,
                       const int64_t* pm, const int64_t* pn, int64_t* acc,
                       float* f, uint16_t* y) {
    for (int64_t i = 0; i < npts; ++i)
        if (pm[i] < 0 || pm[i] >= m_rows || pn[i] < 0 || pn[i] >= n_rows) return ORACLE_ERR_ARG;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t m = pm[i], n = pn[i];
        int64_t sum = 0;
        for (int64_t j = 0; j < k; ++j)
            sum += (int64_t)qx[m * k + j] * (int64_t)qw[n * k + j];
        acc[i] = sum;
        int rc = w8a8_point(sum, sx[m], sw[n], bias, n, &f[i], &y[i]);
        if (rc) {
#pragma omp atomic write
            err = rc;
        }
    }
    return err;
}

/* Weight-only W8A16 as dequantize-then-matmul in fp64 [W8A16][Q]:
 *   y[m,n] = sum_k (s[n] * q[n,k]) * x[m,k]. */
int oracle_w8a16(const uint16_t* x, const int8_t* q, const float* s,
                 int64_t m_rows, int64_t n_rows, int64_t k, double* y) {
    if (m_rows < 0 || n_rows < 0 || k < 0) return ORACLE_ERR_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < m_rows; ++m)
        for (int64_t n = 0; n < n_rows; ++n) {
            double sum = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                double w = (double)s[n] * (double)q[n * k + j];
                sum += w * (double)widen_bf16(x[m * k + j]);
            }
            y[m * n_rows + n] = sum;
        }
    return ORACLE_OK;
}

/* W8A16 at chosen output points. */
int oracle_w8a16_points(const uint16_t* x, const int8_t* q, const float* s,
                        int64_t m_rows, int64_t n_rows, int64_t k, int64_t npts,
                        const int64_t* pm, const int64_t* pn, double* y) {
    for (int64_t i = 0; i < npts; ++i)
        if (pm[i] < 0 || pm[i] >= m_rows || pn[i] < 0 || pn[i] >= n_rows) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t m = pm[i], n = pn[i];
        double sum = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            double w = (double)s[n] * (double)q[n * k + j];
            sum += w * (double)widen_bf16(x[m * k + j]);
        }
        y[i] = sum;
    }
    return ORACLE_OK;
}

/* Grouped W8A16 over experts [MOE]: rows off[e] .. off[e+1] of x go through
 * expert e's weights q[e] ([N, K]) and scales s[e] ([N]).  The offsets must
 * start at 0, never decrease, and end at t_total. */
int oracle_grouped_w8a16(const uint16_t* x, const int32_t* off, int64_t experts,
                         const int8_t* q, const float* s, int64_t t_total,
                         int64_t n_rows, int64_t k, double* y) {
    if (experts < 0 || t_total < 0 || n_rows < 0 || k < 0) return ORACLE_ERR_ARG;
    if (off[0] != 0 || off[experts] != t_total) return ORACLE_ERR_OFFSETS;
    for (int64_t e = 0; e < experts; ++e)
        if (off[e + 1] < off[e]) return ORACLE_ERR_OFFSETS;
    for (int64_t e = 0; e < experts; ++e) {
        const int8_t* qe = q + e * n_rows * k;
        const float* se = s + e * n_rows;
#pragma omp parallel for collapse(2) schedule(static)
        for (int64_t r = off[e]; r < off[e + 1]; ++r)
            for (int64_t n = 0; n < n_rows; ++n) {
                double sum = 0.0;
                for (int64_t j = 0; j < k; ++j) {
                    double w = (double)se[n] * (double)qe[n * k + j];
                    sum += w * (double)widen_bf16(x[r * k + j]);
                }
                y[r * n_rows + n] = sum;
            }
    }
    return ORACLE_OK;
}

/* binary32 -> bf16 (RNE) over an array; exposed so that tests can pin it. */
void oracle_narrow_bf16(const float* f, int64_t count, uint16_t* out) {
    for (int64_t i = 0; i < count; ++i) out[i] = narrow_bf16_rne(f[i]);
}
