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

/* ================================================================ FP8 E4M3
 * [FP8] "Day 6", The mechanism, block 2: FP8 E4M3 is one sign bit, four
 * exponent bits and three mantissa bits, a logarithmic grid dense near zero
 * whose largest value is 448.  Block 1 defines the stored tensor as
 * q = clamp(round(w / s)) with s = absmax / (largest representable value),
 * here s = absmax / 448; block 5 and the FP8_DYNAMIC recipe apply it per
 * output channel to weights and per token, at run time, to activations.
 *
 * Code layout (the E4M3 variant without infinities): bits s eeee mmm,
 * exponent bias 7; e = 0 holds the subnormals (m / 8) * 2^-6; e = 1 .. 15
 * hold (1 + m / 8) * 2^(e - 7), except s.1111.111, which is NaN.  So the
 * non-negative finite codes 0x00 .. 0x7e are increasing in value, from 0 to
 * 448.  Readings: "round" is round to nearest with ties to the even code
 * (even mantissa), "clamp" saturates beyond 448 to +-448, the sign of a value
 * that rounds to zero is kept, and an all-zero row stores s = 1 (as for
 * int8).
 */

float oracle_fp8_decode(uint8_t c) {
    int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    float mag = (e == 0) ? ldexpf((float)m / 8.0f, -6) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return (c & 0x80) ? -mag : mag;
}

/* Nearest E4M3 code of a finite v: the largest non-negative code whose value
 * does not exceed |v| is found by bisection over the increasing codes
 * 0x00 .. 0x7e, then the nearer of it and the next code is taken (ties to
 * the even code); beyond 448 the result saturates to 0x7e. */
uint8_t oracle_fp8_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7e;
    int lo = 0, hi = 0x7e; /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if ((double)oracle_fp8_decode((uint8_t)mid) <= a) lo = mid; else hi = mid;
    }
    double below = a - (double)oracle_fp8_decode((uint8_t)lo);
    double above = (double)oracle_fp8_decode((uint8_t)hi) - a;
    int c = (below < above) ? lo : (above < below) ? hi : ((lo & 1) == 0 ? lo : hi);
    return sign | (uint8_t)c;
}

void oracle_fp8_encode_array(const float* v, int64_t count, uint8_t* out) {
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_fp8_encode(v[i]);
}

void oracle_fp8_decode_array(const uint8_t* c, int64_t count, float* out) {
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_fp8_decode(c[i]);
}

/* Per-row FP8 quantization [FP8]: a = max |v| (fp32), s = a / 448 in fp32
 * (1 if a == 0), q = encode(v / s) with one IEEE fp32 division. */
int oracle_quant_rows_fp8(const uint16_t* src, int64_t rows, int64_t k, uint8_t* q, float* s) {
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
        float scale = (a == 0.0f) ? 1.0f : a / 448.0f;
        s[r] = scale;
        for (int64_t j = 0; j < k; ++j) q[r * k + j] = oracle_fp8_encode(widen_bf16(row[j]) / scale);
    }
    return ORACLE_OK;
}

/* FP8 W8A8 at chosen output points [FP8][W8A8]:
 *   y = (sum_k dec(qx[m,k]) * dec(qw[n,k])) * sx[m] * sw[n] (+ bias[n]).
 * The sum is exact in fp64: every product of two E4M3 values is a multiple
 * of 2^-18 below 2^18, so a sum of at most 2^17 of them is a multiple of
 * 2^-18 below 2^35, which 53 bits hold.  The scales and bias are applied in
 * fp64; the result is the exact value the GPU's bf16 output approximates. */
int oracle_w8a8_fp8_points(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw,
                           const uint16_t* bias, int64_t m_rows, int64_t n_rows, int64_t k,
                           int64_t npts, const int64_t* pm, const int64_t* pn, double* acc, double* y) {
    if (k > ((int64_t)1 << 17)) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < npts; ++i)
        if (pm[i] < 0 || pm[i] >= m_rows || pn[i] < 0 || pn[i] >= n_rows) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t m = pm[i], n = pn[i];
        double sum = 0.0;
        for (int64_t j = 0; j < k; ++j)
            sum += (double)oracle_fp8_decode(qx[m * k + j]) * (double)oracle_fp8_decode(qw[n * k + j]);
        acc[i] = sum;
        double f = sum * (double)sx[m] * (double)sw[n];
        if (bias) f += (double)widen_bf16(bias[n]);
        y[i] = f;
    }
    return ORACLE_OK;
}

/* ================================================================ W4A16, g128
 * [G128] "Day 6", The mechanism, block 1: a W4A16-g128 tensor is int4 codes
 * plus one bf16 scale per 128 weights along the input dimension, with
 * q = clamp(round(w / s)) and s = absmax(group) / (largest code, 7 on the
 * symmetric int4 grid); block 5: the codes are dequantized inside the kernel
 * and the product runs on bf16 math.
 * Readings: the scale is computed in fp32 and stored rounded to bf16 (RNE);
 * the codes divide by the stored scale, so that w ~ s * q holds for the s a
 * kernel reads; codes are clamped to [-7, 7]; an all-zero group stores s = 1
 * and zero codes; ties go to even.  Storage: two codes per byte, even k in
 * the low nibble and odd k in the high nibble, 4-bit two's complement;
 * scales [rows, k / 128].  A nonzero group whose scale rounds to zero in
 * bf16 (absmax below about 2^-131) is outside the contract.
 */
#define ORACLE_ERR_RANGE 5

int oracle_quant_w4_g128(const uint16_t* src, int64_t rows, int64_t k, uint8_t* packed, uint16_t* scale) {
    if (rows < 0 || k < 0 || k % 128 != 0) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < rows * k; ++i)
        if (!isfinite(widen_bf16(src[i]))) return ORACLE_ERR_NONFINITE;
    int err = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < k / 128; ++g) {
            const uint16_t* grp = src + r * k + g * 128;
            float a = 0.0f;
            for (int j = 0; j < 128; ++j) {
                float av = fabsf(widen_bf16(grp[j]));
                if (av > a) a = av;
            }
            uint16_t sb = (a == 0.0f) ? narrow_bf16_rne(1.0f) : narrow_bf16_rne(a / 7.0f);
            float sv = widen_bf16(sb);
            if (sv == 0.0f) {
#pragma omp atomic write
                err = ORACLE_ERR_RANGE;
            }
            scale[r * (k / 128) + g] = sb;
            for (int j = 0; j < 128; j += 2) {
                int c[2];
                for (int h = 0; h < 2; ++h) {
                    float t = (sv == 0.0f) ? 0.0f : widen_bf16(grp[j + h]) / sv;
                    float cr = round_half_even(t);
                    if (cr > 7.0f) cr = 7.0f;
                    if (cr < -7.0f) cr = -7.0f;
                    c[h] = (int)cr;
                }
                packed[r * (k / 2) + (g * 128 + j) / 2] = (uint8_t)((c[0] & 15) | ((c[1] & 15) << 4));
            }
        }
    }
    return err;
}

/* The signed code of weight (n, j) from the packed storage. */
static int w4_code(const uint8_t* packed, int64_t k, int64_t n, int64_t j) {
    uint8_t byte = packed[n * (k / 2) + j / 2];
    int nib = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
    return nib >= 8 ? nib - 16 : nib;
}

void oracle_w4_unpack(const uint8_t* packed, int64_t rows, int64_t k, int8_t* codes) {
    for (int64_t n = 0; n < rows; ++n)
        for (int64_t j = 0; j < k; ++j) codes[n * k + j] = (int8_t)w4_code(packed, k, n, j);
}

/* W4A16 as dequantize-then-matmul in fp64 [G128][W8A16]:
 *   y[m,n] = sum_k (s[n, k / 128] * q[n,k]) * x[m,k]. */
int oracle_w4a16(const uint16_t* x, const uint8_t* packed, const uint16_t* scale, int64_t m_rows,
                 int64_t n_rows, int64_t k, double* y) {
    if (m_rows < 0 || n_rows < 0 || k < 0 || k % 128 != 0) return ORACLE_ERR_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < m_rows; ++m)
        for (int64_t n = 0; n < n_rows; ++n) {
            double sum = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                double w = (double)widen_bf16(scale[n * (k / 128) + j / 128]) * (double)w4_code(packed, k, n, j);
                sum += w * (double)widen_bf16(x[m * k + j]);
            }
            y[m * n_rows + n] = sum;
        }
    return ORACLE_OK;
}

/* ================================================================ MoE expert MLP
 * [MOE] "Phase 5a: int8 weight-only quantization", Summary: the quantized
 * grouped GEMM serves the MoE layer of deepseek-moe-16b, whose experts each
 * hold a fused gate/up projection and a down projection.  The layer around
 * it, as the benchmark configuration states it: gate logits -> softmax ->
 * top-6 routed experts per token, plus two shared experts that see every
 * token.  Readings (the pages give no formulas for these steps): the
 * expert MLP is down(silu(gate(x)) * up(x)) with the gate rows first in the
 * fused projection; a token's output is the sum of its routed experts'
 * outputs weighted by their softmax probabilities (over all routed experts,
 * not renormalised over the six) plus its shared experts' outputs with
 * weight 1; top-k picks the largest logits (the softmax is increasing in the
 * logit), the lower expert index first among equal logits.
 */

/* Routing of T tokens over E routed experts plus `shared` shared experts.
 * Outputs: sel [T, topk] routed expert ids in decreasing logit order;
 * prob [T, topk] their softmax probabilities (fp64); offsets [E + shared + 1];
 * row_token [T * (topk + shared)] the token of each grouped row (rows grouped
 * by expert, tokens increasing within an expert); token_row [T, topk + shared]
 * the grouped row of each (token, slot). */
int oracle_moe_route(const float* logits, int64_t T, int64_t E, int64_t topk, int64_t shared,
                     int32_t* sel, double* prob, int32_t* offsets, int32_t* row_token, int32_t* token_row) {
    if (T < 0 || E <= 0 || E > 4096 || topk <= 0 || topk > E || shared < 0) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < T * E; ++i)
        if (!isfinite(logits[i])) return ORACLE_ERR_NONFINITE;
    int64_t S = topk + shared;
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        double mx = -INFINITY;
        for (int64_t e = 0; e < E; ++e)
            if ((double)l[e] > mx) mx = (double)l[e];
        double den = 0.0;
        for (int64_t e = 0; e < E; ++e) den += exp((double)l[e] - mx);
        unsigned char taken[4096];
        memset(taken, 0, (size_t)E);
        for (int64_t s = 0; s < topk; ++s) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e; /* strict: lower index wins ties */
            taken[best] = 1;
            sel[t * topk + s] = (int32_t)best;
            prob[t * topk + s] = exp((double)l[best] - mx) / den;
        }
    }
    /* rows grouped by expert, tokens in increasing order within an expert */
    int64_t row = 0;
    for (int64_t e = 0; e < E + shared; ++e) {
        offsets[e] = (int32_t)row;
        for (int64_t t = 0; t < T; ++t) {
            int64_t slot = -1;
            if (e < E) {
                for (int64_t s = 0; s < topk; ++s)
                    if (sel[t * topk + s] == e) slot = s;
            } else {
                slot = topk + (e - E);
            }
            if (slot >= 0) {
                row_token[row] = (int32_t)t;
                token_row[t * S + slot] = (int32_t)row;
                ++row;
            }
        }
    }
    offsets[E + shared] = (int32_t)row;
    return ORACLE_OK;
}

/* SiLU-gated product of a fused gate/up output [MOE]: gu [rows, 2I] holds
 * the gate in columns 0 .. I-1 and the up projection in I .. 2I-1;
 * h = silu(g) * u with silu(g) = g / (1 + exp(-g)), in fp64. */
void oracle_silu_mul(const double* gu, int64_t rows, int64_t inter, double* h) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < inter; ++j) {
            double g = gu[r * 2 * inter + j];
            double u = gu[r * 2 * inter + inter + j];
            h[r * inter + j] = g / (1.0 + exp(-g)) * u;
        }
}

/* Weighted combine [MOE]: out[t, :] = sum_s w[t, s] * yd[token_row[t, s], :],
 * slots in order, fp64. */
void oracle_moe_combine(const double* yd, const int32_t* token_row, const double* w, int64_t T, int64_t S,
                        int64_t H, double* out) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            double sum = 0.0;
            for (int64_t s = 0; s < S; ++s) sum += w[t * S + s] * yd[(int64_t)token_row[t * S + s] * H + h];
            out[t * H + h] = sum;
        }
}
