/*
 * oracle.h -- scalar f64 CPU oracle for RMSNorm, the post-norm-then-add shape
 * and the dual-epsilon sandwich tail.
 *
 * TEST INFRASTRUCTURE ONLY.  This code is the reference that the CUDA path is
 * checked against; it is never part of the product path.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, helper or constant with the CUDA library.
 *
 * Sources (page titles and sections):
 *   [P1] "Chapter 12 -- RMSNorm and the dual-epsilon sandwich", section 12.1
 *        (definition), 12.3 (worked example), 12.4.3 (the dual-eps tail:
 *        hidden += rms_norm(src, eps1) * w1; output = rms_norm(hidden, eps2) * w2),
 *        12.4.4 (the split route's f32 publication boundary between the norms),
 *        12.7 (the cross-vendor seam: the weightless norm materialised in F16,
 *        the learned-weight multiply applied as a second F16 operation).
 *   [P4] "RMSNorm Layer - Root Mean Square Normalization" (Hesper API docs),
 *        rmsNormThenAddKernel / rmsNormThenAddBatchKernel:
 *        output = RMSNorm(layer_out) * scale + residual;
 *        rmsNormThenAddThenBroadcastScaleKernel: the same times out_scale[0];
 *        residualAddRmsNormKernel: residualOut = a + b,
 *        output = RMSNorm(residualOut) * scale;
 *        fusedRMSNormQ8_1Kernel: the norm followed by per-32-block
 *        d = amax/127, q = round(x/d), s = 0.
 *
 * Layout: every row operand is a contiguous row-major [rows x n] array of
 * double, row r at base + r*n; gamma is [n] and shared by all rows.  Inputs
 * of narrower types (f32, bf16) are widened to double by the caller, which is
 * exact.  Accumulation is a plain sequential double sum in column order.
 *
 * Parity status: every function below is pinned by CPU tests against the
 * pages' worked example, closed forms, a library routine in f64, exact
 * rational arithmetic on tiny inputs and structural invariants.
 */
#ifndef MRN_ORACLE_H
#define MRN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* y[r,j] = x[r,j] * (1 / sqrt(mean_j(x[r,:]^2) + eps)) * gamma[j]      [P1 12.1] */
void oracle_rmsnorm(const double *x, const double *gamma, double *y,
                    int64_t rows, int64_t n, double eps);

/* out[r,j] = RMSNorm(x[r,:]; eps)[j] * gamma[j] + residual[r,j]      [P4 ThenAdd] */
void oracle_rmsnorm_then_add(const double *x, const double *gamma,
                             const double *residual, double *out,
                             int64_t rows, int64_t n, double eps);

/*
 * Dual-epsilon sandwich tail                                   [P1 12.4.3]
 *   out_stream = RMSNorm(block_out; eps_post) * gamma_post + residual
 *   normed     = RMSNorm(out_stream; eps_pre) * gamma_pre
 * When stream_bf16 is non-zero, out_stream is rounded to bf16 (round to
 * nearest, ties to even) before it is stored and before the second norm
 * reads it: the stored stream is what the second norm sees, as on the split
 * route's publication boundary [P1 12.4.4].
 */
void oracle_norm_residual_norm(const double *block_out, const double *residual,
                               const double *gamma_post, const double *gamma_pre,
                               double *out_stream, double *normed,
                               int64_t rows, int64_t n,
                               double eps_post, double eps_pre, int stream_bf16);

/*
 * Residual add, then RMSNorm of the sum            [P4 residualAddRmsNormKernel]
 *   residual_out = a + b
 *   normed       = RMSNorm(residual_out; eps) * gamma
 * With sum_bf16 non-zero the sum is rounded to bf16 before it is stored and
 * normed, as the sandwich's stream is.
 */
void oracle_add_rmsnorm(const double *a, const double *b, const double *gamma,
                        double *residual_out, double *normed,
                        int64_t rows, int64_t n, double eps, int sum_bf16);

/*
 * Post norm, residual add, then a broadcast scalar   [P4 rmsNormThenAddThenBroadcastScaleKernel]
 *   out = (RMSNorm(x; eps) * gamma + residual) * out_scale
 */
void oracle_rmsnorm_then_add_scale(const double *x, const double *gamma,
                                   const double *residual, double out_scale, double *out,
                                   int64_t rows, int64_t n, double eps);

/*
 * RMSNorm fused with Q8_1 block quantisation      [P4 fusedRMSNormQ8_1Kernel]
 *   x_normed_j = x_j * gamma_j * inv_rms            (the page's product order)
 *   per block of 32 elements: amax = max |x_normed|, d = amax / 127,
 *   qreal_j = x_normed_j / d   (0 for every element when d == 0),
 *   q_j = qreal_j rounded half to even, clamped to [-128, 127]
 * n must be a multiple of 32.  Outputs: d [rows x n/32], qreal [rows x n]
 * (the value before rounding, so a test can see how close a code is to a
 * rounding boundary) and q [rows x n].
 */
void oracle_rmsnorm_q8_1(const double *x, const double *gamma, int64_t rows, int64_t n,
                         double eps, double *d, double *qreal, int8_t *q);
/* The code of one quotient: nearest integer, ties to even, clamped to int8. */
int oracle_q8_round(double qreal);

/*
 * Split-norm seam: the rounding point between the weightless norm and the
 * weight multiply kept                                   [P1 12.7, cross-vendor seam]
 *   u[r,j] = round_T(x[r,j] * inv_rms(x[r,:]; eps))     weightless norm, stored in T
 *   y[r,j] = round_T(u[r,j] * gamma[j])                  weight multiply as a T operation
 * T is IEEE binary16 when seam_bf16 == 0, bf16 otherwise; round_T is round to
 * nearest, ties to even.  gamma holds values of T (the caller widens the
 * patterns).  u and y receive the exact values of their T patterns.  The
 * product u * gamma of two T values is exact in double, so y is the
 * correctly rounded T product.
 */
void oracle_rmsnorm_seam(const double *x, const double *gamma, double *u, double *y,
                         int64_t rows, int64_t n, double eps, int seam_bf16);

/* IEEE binary16 (1 sign, 5 exponent, 10 fraction bits): round a double to the
 * nearest (ties to even), and widen a pattern exactly. */
uint16_t oracle_f16_from_double(double v);
double oracle_double_from_f16(uint16_t bits);

/* Round a double to the nearest bf16 (ties to even); returns the bit pattern. */
uint16_t oracle_bf16_from_double(double v);
/* Exact value of a bf16 bit pattern. */
double oracle_double_from_bf16(uint16_t bits);
/* Array forms of the two conversions above. */
void oracle_bf16_round_array(const double *v, uint16_t *bits, int64_t count);
void oracle_bf16_widen_array(const uint16_t *bits, double *v, int64_t count);

#ifdef __cplusplus
}
#endif

#endif /* MRN_ORACLE_H */
