/*
 * mxq_oracle.c -- scalar CPU oracle for OCP-MX block-scaled quantization.
 *
 * TEST INFRASTRUCTURE ONLY (see mxq_oracle.h).  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load this code; the CUDA
 * library never does, and the two share no source.
 *
 * Build: plain C99, -O2 -ffp-contract=off, no fast-math, no SIMD intrinsics,
 * so every float operation below is one IEEE-754 operation in the stated
 * precision.
 *
 * What is computed, and where it comes from:
 *
 *  MXFP8 (kernel families "MXFP8 generic quantize", "MXFP8 specialized
 *  cast-only" and "MXFP8 gated" in TransformerEngine PR #3291 "Fix pointer
 *  arithmatic to generate correct LDS/STS instructions", results tables;
 *  colwise "dim1" cast of torchao PR #12 "Multiply with inverse scale in loop
 *  instead of dividing").  Neither page writes the arithmetic out; the rule
 *  this library implements is:
 *    per block of 32 values y (1x32 along K for rowwise, 32x1 along M for
 *    colwise):  a = max |y|;  e = clamp(floor(log2 a) - 8, -127, 127), with
 *    a = 0 giving the code 0;  scale byte = e + 127 (E8M0);  every element
 *    becomes E4M3(y * 2^-e) with round-to-nearest-even and saturation to
 *    +-448.  8 is the exponent of the largest E4M3 binade (448 = 1.75*2^8).
 *    The multiply by 2^-e is the "inverse scale" of torchao PR #12 (its
 *    rationale section): one reciprocal per block, then a multiply per
 *    element; here the reciprocal is an exact power of two.
 *    With ORC_SCALE_RCEIL the shared exponent follows the ceil-style rule
 *    instead: e = ceil(log2(a / 448)), the smallest power of two for which
 *    no element of the block exceeds 448 (so nothing saturates), clamped
 *    the same way.
 *
 *  Activations (TE PR #3291, "MXFP8 generic" fusion "gelu" and "MXFP8 gated"
 *  fusion "swiglu"): y is computed in double and rounded once to fp32, then
 *  quantized as above.  GELU is the tanh form
 *    0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)));
 *  SwiGLU is silu(g) * u with silu(g) = g / (1 + e^-g); GeGLU (gated kernel
 *  fusion "geglu") is gelu_tanh(g) * u.
 *  Backward fusions (generic kernel fusions "dgelu", "dsilu", "dbias_dgelu";
 *  gated kernel fusion "dswiglu", and its GeGLU counterpart): with grad the
 *  incoming gradient, y = grad * act'(x) (dbias = column sums of y); for the
 *  gated forms the output is [d gate | d up] = [grad * up * act'(gate) |
 *  grad * act(gate)], 2N columns.  The derivatives are the closed forms
 *  of the two functions above, evaluated in double.
 *
 *  dbias (TE PR #3291, fusion "dbias"): dbias[k] = sum over m of x[m][k],
 *  the exact sum rounded to fp32 (compensated summation in double).
 *
 *  NVFP4 (TE PR #3291, "NVFP4 quantize-transpose" kernel family; the 1D
 *  1x16 variant named in its "Patched but not measurable" section).  Neither
 *  page gives the recipe; the reading implemented here, every step one fp32
 *  IEEE operation in this order:
 *    G = A / 2688 (A = tensor amax, 2688 = 448 * 6);
 *    per block of 16: b = block amax; s = E4M3((b / 6) / G);
 *    d = value(s) * G;  inv = (s == 0 or d == 0) ? 0 : 1 / d, replaced by
 *    the largest finite float if 1 / d overflows;
 *    every element becomes E2M1(x * inv), round-to-nearest-even, saturating
 *    to +-6;  A = 0 gives G = 0 and every scale 0.
 *  The 2D variant (TE PR #3291, results table "NVFP4 2D quantize-transpose
 *  kernel", fusion "nvfp42d") takes b over a 16x16 block instead, the rest
 *  unchanged; its scale bytes keep the 1D layouts, each repeated over the
 *  block's 16 rows (rowwise) or 16 columns (transposed).
 *
 *  NaN and infinite inputs are outside the contract; the choices made for
 *  them below are documented but not checked against the GPU.
 */
#include "mxq_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Rounding helper                                                          */
/* ------------------------------------------------------------------------ */

/* Round a non-negative double to the nearest integer, ties to even.
 * q - floor(q) is exact for q < 2^52. */
static double rne_nonneg(double q) {
    double f = floor(q);
    double frac = q - f;
    if (frac > 0.5) return f + 1.0;
    if (frac < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                           */
/* ------------------------------------------------------------------------ */

double orc_bf16_decode(uint16_t bits) {
    int sign = bits >> 15;
    int e = (bits >> 7) & 0xFF;
    int m = bits & 0x7F;
    double mag;
    if (e == 0xFF) mag = m ? NAN : INFINITY;
    else if (e == 0) mag = ldexp((double)m, -133);          /* m * 2^-7 * 2^-126 */
    else mag = ldexp(128.0 + m, e - 127 - 7);                /* (1 + m/128) 2^(e-127) */
    return sign ? -mag : mag;
}

/* E4M3 value -> code.  Round to nearest, ties to even mantissa; magnitudes
 * above 448 saturate to 448 (code 0x7E); the sign is kept, so -0 and
 * negative values that round to zero give 0x80. */
uint8_t orc_e4m3_encode(double v) {
    uint8_t s = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (isnan(v)) return s | 0x7F;
    if (a >= 448.0) return s | 0x7E;
    if (a < 0x1p-6) {
        /* Subnormal binade: values n * 2^-9, n = 0..7.  n = 8 is the
         * smallest normal 2^-6, whose code is also 8 (exponent field 1). */
        double n = rne_nonneg(ldexp(a, 9));
        return s | (uint8_t)n;
    }
    int ex;
    frexp(a, &ex);             /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;            /* a in [2^E, 2^(E+1)), E in [-6, 8] */
    double n = rne_nonneg(ldexp(a, 3 - E));   /* 8 significand steps per binade */
    if (n == 16.0) {           /* rounded up into the next binade */
        n = 8.0;
        E += 1;
    }
    int code = ((E + 7) << 3) | ((int)n - 8);
    if (code > 0x7E) code = 0x7E;   /* unreachable for a < 448; guard only */
    return s | (uint8_t)code;
}

double orc_e4m3_decode(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(8.0 + m, e - 7 - 3);
    return sign ? -mag : mag;
}

/* E2M1 value -> 4-bit code, round to nearest, ties to even mantissa,
 * saturating to 6; sign kept (-0 -> 0x8).  NaN saturates (documented). */
uint8_t orc_e2m1_encode(double v) {
    uint8_t s = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    if (isnan(v) || a >= 6.0) return s | 0x7;
    if (a < 1.0) {
        /* Subnormal binade: 0 and 0.5; n = 2 is the smallest normal 1.0. */
        double n = rne_nonneg(a * 2.0);
        return s | (uint8_t)n;
    }
    int ex;
    frexp(a, &ex);
    int E = ex - 1;                            /* 0, 1 or 2 */
    double n = rne_nonneg(ldexp(a, 1 - E));    /* 2 significand steps per binade */
    if (n == 4.0) {
        n = 2.0;
        E += 1;
    }
    int code = ((E + 1) << 1) | ((int)n - 2);
    if (code > 7) code = 7;
    return s | (uint8_t)code;
}

double orc_e2m1_decode(uint8_t code) {
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 0x3;
    int m = code & 0x1;
    double mag = (e == 0) ? 0.5 * m : ldexp(2.0 + m, e - 1 - 1);
    return sign ? -mag : mag;
}

/* MX shared scale: floor(log2 amax) - 8, clamped to [-127, 127], biased by
 * 127.  amax = 0 gives 0.  floor(log2 a) is read off frexp exactly. */
uint8_t orc_e8m0_code(double amax) {
    if (isnan(amax)) return 0xFF;              /* E8M0 NaN; outside the contract */
    if (!(amax > 0.0)) return 0;
    if (isinf(amax)) return 0xFE;
    int ex;
    frexp(amax, &ex);
    int e = (ex - 1) - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

void orc_e4m3_encode_array(const double* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

void orc_e2m1_encode_array(const double* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_encode(v[i]);
}

/* The ceil-style rule: e = ceil(log2(amax / 448)), the smallest power of two
 * for which no element of the block exceeds the E4M3 maximum 448, clamped
 * to [-127, 127]; amax = 0 gives code 0. */
uint8_t orc_e8m0_code_rceil(double amax) {
    if (isnan(amax)) return 0xFF;
    if (!(amax > 0.0)) return 0;
    if (isinf(amax)) return 0xFE;
    double e = ceil(log2(amax / 448.0));
    if (e < -127.0) e = -127.0;
    if (e > 127.0) e = 127.0;
    return (uint8_t)((int)e + 127);
}

void orc_e8m0_code_rceil_array(const double* amax, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e8m0_code_rceil(amax[i]);
}

void orc_e8m0_code_array(const double* amax, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e8m0_code(amax[i]);
}

/* ------------------------------------------------------------------------ */
/* Activations                                                              */
/* ------------------------------------------------------------------------ */

static const double ORC_PI = 3.14159265358979323846264338327950288;

float orc_gelu_tanh(float x) {
    double xd = (double)x;
    double u = sqrt(2.0 / ORC_PI) * (xd + 0.044715 * xd * xd * xd);
    /* 1 + tanh(u); for u < 0 the sum cancels in double, so use the exact
     * identity 1 + tanh(u) = 2 e^(2u) / (1 + e^(2u)) there. */
    double one_plus_tanh;
    if (u >= 0.0) {
        one_plus_tanh = 1.0 + tanh(u);
    } else {
        double t = exp(2.0 * u);
        one_plus_tanh = 2.0 * t / (1.0 + t);
    }
    return (float)(0.5 * xd * one_plus_tanh);
}

float orc_swiglu(float gate, float up) {
    double g = (double)gate;
    double silu = g / (1.0 + exp(-g));
    return (float)(silu * (double)up);
}

/* gelu_tanh(x) and its derivative in double.  With u = c (x + a x^3),
 * s = e^(-2|u|):  tanh|u| = (1 - s) / (1 + s), so 1 + tanh(u) is 2 / (1 + s)
 * for u >= 0 and 2 s / (1 + s) for u < 0, and 1 - tanh(u)^2 = 4 s / (1 + s)^2
 * (no cancellation on either side).
 *   d/dx 0.5 x (1 + tanh u) = 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) c (1 + 3 a x^2). */
static void gelu_tanh_d(double x, double* value, double* deriv) {
    const double c = sqrt(2.0 / ORC_PI), a = 0.044715;
    double u = c * (x + a * x * x * x);
    double s = exp(-2.0 * fabs(u));
    double one_plus_tanh = (u >= 0.0) ? 2.0 / (1.0 + s) : 2.0 * s / (1.0 + s);
    double sech2 = 4.0 * s / ((1.0 + s) * (1.0 + s));
    if (value) *value = 0.5 * x * one_plus_tanh;
    if (deriv) *deriv = 0.5 * one_plus_tanh + 0.5 * x * sech2 * c * (1.0 + 3.0 * a * x * x);
}

/* silu(x) = x sigma(x) and its derivative sigma(x) (1 + x sigma(-x)), in
 * double (sigma(-x) = 1 - sigma(x) taken directly, no cancellation). */
static void silu_d(double x, double* value, double* deriv) {
    double sp = 1.0 / (1.0 + exp(-x));
    double sm = 1.0 / (1.0 + exp(x));
    if (value) *value = x * sp;
    if (deriv) *deriv = sp * (1.0 + x * sm);
}

static void act_d(int act, double x, double* value, double* deriv) {
    if (act == ORC_ACT_GELU_TANH) gelu_tanh_d(x, value, deriv);
    else silu_d(x, value, deriv);
}

float orc_geglu(float gate, float up) {
    double v;
    gelu_tanh_d((double)gate, &v, NULL);
    return (float)(v * (double)up);
}

float orc_dgelu_tanh(float x) {
    double d;
    gelu_tanh_d((double)x, NULL, &d);
    return (float)d;
}

float orc_dsilu(float x) {
    double d;
    silu_d((double)x, NULL, &d);
    return (float)d;
}

/* ------------------------------------------------------------------------ */
/* MXFP8                                                                    */
/* ------------------------------------------------------------------------ */

/* Quantize one MX block of 32 fp32 values.  y[i * ys] are the values,
 * q[i * qs] receive the E4M3 codes, *scale the E8M0 code. */
static void mx_block(const float* y, int64_t ys, uint8_t* q, int64_t qs, uint8_t* scale,
                     int rceil) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
        double a = fabs((double)y[i * ys]);
        if (a > amax) amax = a;
    }
    uint8_t code = rceil ? orc_e8m0_code_rceil(amax) : orc_e8m0_code(amax);
    int e = (int)code - 127;
    *scale = code;
    for (int i = 0; i < 32; ++i) {
        /* y * 2^-e: exact in double for every fp32 y and every e. */
        q[i * qs] = orc_e4m3_encode(ldexp((double)y[i * ys], -e));
    }
}

/* Rowwise and colwise MX quantization of a dense fp32 matrix y[M][K]. */
static void mx_quantize_dense(const float* y, int64_t M, int64_t K, int flags,
                              uint8_t* q_row, uint8_t* s_row,
                              uint8_t* q_col, uint8_t* s_col) {
    if (flags & ORC_ROWWISE) {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t kb = 0; kb < K / 32; ++kb)
                mx_block(y + m * K + kb * 32, 1, q_row + m * K + kb * 32, 1,
                         s_row + m * (K / 32) + kb, flags & ORC_SCALE_RCEIL);
    }
    if (flags & ORC_COLWISE) {
        for (int64_t k = 0; k < K; ++k)
            for (int64_t mb = 0; mb < M / 32; ++mb)
                mx_block(y + mb * 32 * K + k, K, q_col + k * M + mb * 32, 1,
                         s_col + k * (M / 32) + mb, flags & ORC_SCALE_RCEIL);
    }
}

/* Compensated (Neumaier) sum of column k of y, rounded to fp32. */
static float column_sum(const float* y, int64_t M, int64_t K, int64_t k) {
    double s = 0.0, c = 0.0;
    for (int64_t m = 0; m < M; ++m) {
        double v = (double)y[m * K + k];
        double t = s + v;
        if (fabs(s) >= fabs(v)) c += (s - t) + v;
        else c += (v - t) + s;
        s = t;
    }
    return (float)(s + c);
}

int orc_mx_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                    int flags, int act,
                    uint8_t* q_row, uint8_t* s_row,
                    uint8_t* q_col, uint8_t* s_col, float* dbias) {
    if (!x || M < 0 || K < 0 || ldx < K) return -1;
    if ((M % 32) || (K % 32)) return -1;
    if (act != ORC_ACT_NONE && act != ORC_ACT_GELU_TANH) return -1;
    if (M == 0 || K == 0) {
        if ((flags & ORC_DBIAS) && dbias)
            for (int64_t k = 0; k < K; ++k) dbias[k] = 0.0f;
        return 0;
    }
    float* y = (float*)malloc((size_t)(M * K) * sizeof(float));
    if (!y) return -1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float v = (float)orc_bf16_decode(x[m * ldx + k]);   /* exact */
            y[m * K + k] = (act == ORC_ACT_GELU_TANH) ? orc_gelu_tanh(v) : v;
        }
    mx_quantize_dense(y, M, K, flags, q_row, s_row, q_col, s_col);
    if ((flags & ORC_DBIAS) && dbias)
        for (int64_t k = 0; k < K; ++k) dbias[k] = column_sum(y, M, K, k);
    free(y);
    return 0;
}

int orc_mx_quantize_gated(const uint16_t* x, int64_t M, int64_t N,
                          int64_t ldx, int64_t up_offset, int flags, int act,
                          uint8_t* q_row, uint8_t* s_row,
                          uint8_t* q_col, uint8_t* s_col) {
    if (!x || M < 0 || N < 0 || up_offset < N || ldx < up_offset + N) return -1;
    if ((M % 32) || (N % 32)) return -1;
    if (act != ORC_ACT_SILU && act != ORC_ACT_GELU_TANH) return -1;
    if (M == 0 || N == 0) return 0;
    float* y = (float*)malloc((size_t)(M * N) * sizeof(float));
    if (!y) return -1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            float g = (float)orc_bf16_decode(x[m * ldx + n]);
            float u = (float)orc_bf16_decode(x[m * ldx + up_offset + n]);
            y[m * N + n] = (act == ORC_ACT_SILU) ? orc_swiglu(g, u) : orc_geglu(g, u);
        }
    mx_quantize_dense(y, M, N, flags, q_row, s_row, q_col, s_col);
    free(y);
    return 0;
}

int orc_mx_quantize_swiglu(const uint16_t* x, int64_t M, int64_t N,
                           int64_t ldx, int64_t up_offset, int flags,
                           uint8_t* q_row, uint8_t* s_row,
                           uint8_t* q_col, uint8_t* s_col) {
    return orc_mx_quantize_gated(x, M, N, ldx, up_offset, flags, ORC_ACT_SILU,
                                 q_row, s_row, q_col, s_col);
}

int orc_mx_quantize_dact(const uint16_t* grad, const uint16_t* x, int64_t M, int64_t K,
                         int64_t ldg, int64_t ldx, int flags, int act,
                         uint8_t* q_row, uint8_t* s_row,
                         uint8_t* q_col, uint8_t* s_col, float* dbias) {
    if (!grad || !x || M < 0 || K < 0 || ldg < K || ldx < K) return -1;
    if ((M % 32) || (K % 32)) return -1;
    if (act != ORC_ACT_SILU && act != ORC_ACT_GELU_TANH) return -1;
    if (M == 0 || K == 0) {
        if ((flags & ORC_DBIAS) && dbias)
            for (int64_t k = 0; k < K; ++k) dbias[k] = 0.0f;
        return 0;
    }
    float* y = (float*)malloc((size_t)(M * K) * sizeof(float));
    if (!y) return -1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            double d;
            act_d(act, orc_bf16_decode(x[m * ldx + k]), NULL, &d);
            y[m * K + k] = (float)(orc_bf16_decode(grad[m * ldg + k]) * d);
        }
    mx_quantize_dense(y, M, K, flags, q_row, s_row, q_col, s_col);
    if ((flags & ORC_DBIAS) && dbias)
        for (int64_t k = 0; k < K; ++k) dbias[k] = column_sum(y, M, K, k);
    free(y);
    return 0;
}

int orc_mx_quantize_dgated(const uint16_t* grad, const uint16_t* x, int64_t M, int64_t N,
                           int64_t ldg, int64_t ldx, int64_t up_offset, int flags, int act,
                           uint8_t* q_row, uint8_t* s_row,
                           uint8_t* q_col, uint8_t* s_col) {
    if (!grad || !x || M < 0 || N < 0 || ldg < N || up_offset < N || ldx < up_offset + N)
        return -1;
    if ((M % 32) || (N % 32)) return -1;
    if (act != ORC_ACT_SILU && act != ORC_ACT_GELU_TANH) return -1;
    if (M == 0 || N == 0) return 0;
    const int64_t W = 2 * N;
    float* y = (float*)malloc((size_t)(M * W) * sizeof(float));
    if (!y) return -1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double g = orc_bf16_decode(grad[m * ldg + n]);
            double gate = orc_bf16_decode(x[m * ldx + n]);
            double up = orc_bf16_decode(x[m * ldx + up_offset + n]);
            double v, d;
            act_d(act, gate, &v, &d);
            y[m * W + n] = (float)(g * up * d);       /* d / d gate */
            y[m * W + N + n] = (float)(g * v);        /* d / d up   */
        }
    mx_quantize_dense(y, M, W, flags, q_row, s_row, q_col, s_col);
    free(y);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* NVFP4                                                                    */
/* ------------------------------------------------------------------------ */

float orc_bf16_amax(const uint16_t* x, int64_t M, int64_t K, int64_t ldx) {
    float amax = 0.0f;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf((float)orc_bf16_decode(x[m * ldx + k]));
            if (a > amax) amax = a;
        }
    return amax;
}

/* The E4M3 scale code s of a block with amax b, and the reciprocal inv its
 * elements are multiplied by (the recipe's steps 3-5, each one fp32
 * operation). */
static void nvfp4_scale(float b, float G, uint8_t* scale, float* inv_out) {
    uint8_t s = 0;
    float inv = 0.0f;
    if (G != 0.0f) {
        float sf = (b / 6.0f) / G;
        s = orc_e4m3_encode((double)sf);
        float d = (float)orc_e4m3_decode(s) * G;
        if (s != 0 && d != 0.0f) {
            inv = 1.0f / d;
            if (isinf(inv)) inv = FLT_MAX;
        }
    }
    *scale = s;
    *inv_out = inv;
}

/* One NVFP4 block of 16 values v[i * vs]; writes the E4M3 scale code and
 * the 16 E2M1 codes (one per byte, low nibble). */
static void nvfp4_block(const float* v, int64_t vs, float G, uint8_t* scale, uint8_t* codes) {
    float b = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float a = fabsf(v[i * vs]);
        if (a > b) b = a;
    }
    float inv;
    nvfp4_scale(b, G, scale, &inv);
    for (int i = 0; i < 16; ++i) {
        float p = v[i * vs] * inv;
        codes[i] = orc_e2m1_encode((double)p);
    }
}

/* 2D variant: one scale per 16x16 block (rows 16 mb.., columns 16 kb..),
 * from the amax of its 256 values; every element of the block is quantized
 * with that scale in both outputs, and the scale byte is repeated in each of
 * the block's 16 rows (rowwise scales) and 16 columns (transposed scales). */
static void nvfp4_quantize_2d(const float* v, int64_t M, int64_t K, int flags, float G,
                              uint8_t* q_row, uint8_t* s_row, uint8_t* q_t, uint8_t* s_t) {
    for (int64_t mb = 0; mb < M / 16; ++mb)
        for (int64_t kb = 0; kb < K / 16; ++kb) {
            float b = 0.0f;
            for (int64_t i = 0; i < 16; ++i)
                for (int64_t jj = 0; jj < 16; ++jj) {
                    float a = fabsf(v[(mb * 16 + i) * K + kb * 16 + jj]);
                    if (a > b) b = a;
                }
            uint8_t sc;
            float inv;
            nvfp4_scale(b, G, &sc, &inv);
            for (int64_t i = 0; i < 16; ++i)
                for (int64_t jj = 0; jj < 16; ++jj) {
                    const int64_t m = mb * 16 + i, k = kb * 16 + jj;
                    const uint8_t code = orc_e2m1_encode((double)(v[m * K + k] * inv));
                    if (flags & ORC_ROWWISE) {
                        uint8_t* byte = q_row + m * (K / 2) + k / 2;
                        *byte = (k & 1) ? (uint8_t)((*byte & 0x0F) | (code << 4)) : code;
                    }
                    if (flags & ORC_COLWISE) {
                        uint8_t* byte = q_t + k * (M / 2) + m / 2;
                        *byte = (m & 1) ? (uint8_t)((*byte & 0x0F) | (code << 4)) : code;
                    }
                }
            for (int64_t i = 0; i < 16; ++i) {
                if (flags & ORC_ROWWISE) s_row[(mb * 16 + i) * (K / 16) + kb] = sc;
                if (flags & ORC_COLWISE) s_t[(kb * 16 + i) * (M / 16) + mb] = sc;
            }
        }
}

int orc_nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                       float tensor_amax, int flags, float* global_scale,
                       uint8_t* q_row, uint8_t* s_row,
                       uint8_t* q_t, uint8_t* s_t) {
    if (!x || M < 0 || K < 0 || ldx < K) return -1;
    if ((M % 16) || (K % 16)) return -1;
    float G = tensor_amax / 2688.0f;
    if (global_scale) *global_scale = G;
    if (M == 0 || K == 0) return 0;
    float* v = (float*)malloc((size_t)(M * K) * sizeof(float));
    if (!v) return -1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) v[m * K + k] = (float)orc_bf16_decode(x[m * ldx + k]);
    if (flags & ORC_NVFP4_2D) {
        nvfp4_quantize_2d(v, M, K, flags, G, q_row, s_row, q_t, s_t);
        free(v);
        return 0;
    }
    uint8_t codes[16];
    if (flags & ORC_ROWWISE) {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t kb = 0; kb < K / 16; ++kb) {
                nvfp4_block(v + m * K + kb * 16, 1, G, s_row + m * (K / 16) + kb, codes);
                for (int i = 0; i < 8; ++i)
                    q_row[m * (K / 2) + kb * 8 + i] =
                        (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
            }
    }
    if (flags & ORC_COLWISE) {
        for (int64_t k = 0; k < K; ++k)
            for (int64_t mb = 0; mb < M / 16; ++mb) {
                nvfp4_block(v + mb * 16 * K + k, K, G, s_t + k * (M / 16) + mb, codes);
                for (int i = 0; i < 8; ++i)
                    q_t[k * (M / 2) + mb * 8 + i] =
                        (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
            }
    }
    free(v);
    return 0;
}
