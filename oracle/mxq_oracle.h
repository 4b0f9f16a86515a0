/*
 * mxq_oracle.h -- scalar CPU oracle for OCP-MX block-scaled quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library in
 * fp4_quantization_gb300/) includes, links or calls this code, and this code
 * includes nothing from there.  It exists so the tests, the smoke check and
 * the benchmark's CPU-baseline leg can check the GPU path against a plain,
 * slow, obviously-correct definition.
 *
 * Formats (all little-endian bytes):
 *   bf16  : 1 sign, 8 exponent (bias 127), 7 mantissa bits.
 *   E4M3  : 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinities,
 *           S.1111.111 is NaN, largest finite 448 (S.1111.110), smallest
 *           subnormal 2^-9.
 *   E2M1  : 1 sign, 2 exponent (bias 1), 1 mantissa bit; values
 *           {0, 0.5, 1, 1.5, 2, 3, 4, 6} with sign.
 *   E8M0  : an unsigned byte c meaning the scale 2^(c-127).
 *
 * Layouts used by every function below (row-major, dense):
 *   MX rowwise  codes [M][K]   scales [M][K/32]   (1x32 blocks along K)
 *   MX colwise  codes [K][M]   scales [K][M/32]   (32x1 blocks along M,
 *                                                  stored column-major)
 *   NVFP4 rowwise     codes [M][K/2]  scales [M][K/16]  (1x16 along K)
 *   NVFP4 transposed  codes [K][M/2]  scales [K][M/16]  (16x1 along M)
 *   NVFP4 packing: element 2i in the low nibble, 2i+1 in the high nibble.
 */
#ifndef MXQ_ORACLE_H
#define MXQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_ROWWISE = 1, ORC_COLWISE = 2, ORC_DBIAS = 4, ORC_NVFP4_2D = 16, ORC_SCALE_RCEIL = 64 };
enum { ORC_ACT_NONE = 0, ORC_ACT_GELU_TANH = 1, ORC_ACT_SILU = 2 };

/* Scalar format conversions. */
double  orc_bf16_decode(uint16_t bits);
uint8_t orc_e4m3_encode(double v);      /* RNE, saturate to +-448, keep sign */
double  orc_e4m3_decode(uint8_t code);
uint8_t orc_e2m1_encode(double v);      /* RNE, saturate to +-6, keep sign */
double  orc_e2m1_decode(uint8_t code);
uint8_t orc_e8m0_code(double amax);     /* MX shared-scale rule, see .c */
uint8_t orc_e8m0_code_rceil(double amax);   /* ceil rule (flag ORC_SCALE_RCEIL) */

/* Array forms of the encoders, for brute-force tests. */
void orc_e4m3_encode_array(const double* v, int64_t n, uint8_t* out);
void orc_e2m1_encode_array(const double* v, int64_t n, uint8_t* out);
void orc_e8m0_code_array(const double* amax, int64_t n, uint8_t* out);
void orc_e8m0_code_rceil_array(const double* amax, int64_t n, uint8_t* out);

/* Activations and derivatives evaluated in double and rounded once to fp32. */
float orc_gelu_tanh(float x);
float orc_swiglu(float gate, float up);
float orc_geglu(float gate, float up);
float orc_dgelu_tanh(float x);
float orc_dsilu(float x);

/* MXFP8 quantization of a bf16 matrix x[M][K] (row stride ldx elements).
 * flags: ORC_ROWWISE / ORC_COLWISE select the outputs; ORC_DBIAS writes
 * dbias[k] = sum_m x[m][k] (fp32).  act: ORC_ACT_NONE or ORC_ACT_GELU_TANH.
 * Returns 0, or -1 on a bad argument. */
int orc_mx_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                    int flags, int act,
                    uint8_t* q_row, uint8_t* s_row,
                    uint8_t* q_col, uint8_t* s_col, float* dbias);

/* Gated (SwiGLU) MXFP8: y[m][n] = silu(x[m][n]) * x[m][n + up_offset],
 * n < N, then the same rowwise/colwise quantization of y. */
int orc_mx_quantize_swiglu(const uint16_t* x, int64_t M, int64_t N,
                           int64_t ldx, int64_t up_offset, int flags,
                           uint8_t* q_row, uint8_t* s_row,
                           uint8_t* q_col, uint8_t* s_col);

/* Gated MXFP8 with act ORC_ACT_SILU (SwiGLU) or ORC_ACT_GELU_TANH (GeGLU):
 * y[m][n] = act(gate) * up, gate = x[m][n], up = x[m][n + up_offset]. */
int orc_mx_quantize_gated(const uint16_t* x, int64_t M, int64_t N,
                          int64_t ldx, int64_t up_offset, int flags, int act,
                          uint8_t* q_row, uint8_t* s_row,
                          uint8_t* q_col, uint8_t* s_col);

/* Backward MXFP8: y = grad * act'(x) (act ORC_ACT_GELU_TANH or ORC_ACT_SILU),
 * product in double rounded once; ORC_DBIAS writes the column sums of y. */
int orc_mx_quantize_dact(const uint16_t* grad, const uint16_t* x, int64_t M, int64_t K,
                         int64_t ldg, int64_t ldx, int flags, int act,
                         uint8_t* q_row, uint8_t* s_row,
                         uint8_t* q_col, uint8_t* s_col, float* dbias);

/* Backward gated MXFP8: grad [M][N], x = [gate | up] as for the gated
 * forward; y [M][2N] = [grad * up * act'(gate) | grad * act(gate)]. */
int orc_mx_quantize_dgated(const uint16_t* grad, const uint16_t* x, int64_t M, int64_t N,
                           int64_t ldg, int64_t ldx, int64_t up_offset, int flags, int act,
                           uint8_t* q_row, uint8_t* s_row,
                           uint8_t* q_col, uint8_t* s_col);

/* Largest |x| over a bf16 matrix, as fp32 (exact). */
float orc_bf16_amax(const uint16_t* x, int64_t M, int64_t K, int64_t ldx);

/* NVFP4 quantize + transpose of x[M][K] given the tensor amax A.
 * flags: ORC_ROWWISE / ORC_COLWISE (the latter = transposed output);
 * ORC_NVFP4_2D: one scale per 16x16 block instead of per 1x16 / 16x1 block
 * (same output layouts, each block's scale repeated over its 16 rows or
 * columns). */
int orc_nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                       float tensor_amax, int flags, float* global_scale,
                       uint8_t* q_row, uint8_t* s_row,
                       uint8_t* q_t, uint8_t* s_t);

#ifdef __cplusplus
}
#endif
#endif
