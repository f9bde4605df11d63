/*
 * oracle.c -- scalar f64 CPU oracle (TEST INFRASTRUCTURE ONLY; see oracle.h).
 *
 * Written from the definition on "Chapter 12 -- RMSNorm and the
 * dual-epsilon sandwich", section 12.1:
 *     mean(x^2) = (1/n) sum_j x_j^2
 *     rms       = sqrt(mean(x^2) + eps)
 *     y_i       = x_i / rms * gamma_i
 * The kernels of that chapter compute the reciprocal root once and multiply
 * (x * inv_rms * gamma, section 12.3 step 3); this file does the same in
 * double.  Compile without fast-math and without FMA contraction so that the
 * result is the same on every host.
 */
#include "oracle.h"

#include <math.h>

/* 1 / sqrt(mean of squares + eps) of one row; plain sequential sum. */
static double row_inv_rms(const double *row, int64_t n, double eps)
{
    double sum_sq = 0.0;
    for (int64_t j = 0; j < n; ++j)
        sum_sq += row[j] * row[j];
    double mean_sq = sum_sq / (double)n;
    return 1.0 / sqrt(mean_sq + eps);
}

void oracle_rmsnorm(const double *x, const double *gamma, double *y,
                    int64_t rows, int64_t n, double eps)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * n;
        double *yr = y + r * n;
        double inv_rms = row_inv_rms(xr, n, eps);
        for (int64_t j = 0; j < n; ++j)
            yr[j] = xr[j] * inv_rms * gamma[j];
    }
}

void oracle_rmsnorm_then_add(const double *x, const double *gamma,
                             const double *residual, double *out,
                             int64_t rows, int64_t n, double eps)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * n;
        const double *rr = residual + r * n;
        double *outr = out + r * n;
        double inv_rms = row_inv_rms(xr, n, eps);
        for (int64_t j = 0; j < n; ++j)
            outr[j] = xr[j] * inv_rms * gamma[j] + rr[j];
    }
}

void oracle_norm_residual_norm(const double *block_out, const double *residual,
                               const double *gamma_post, const double *gamma_pre,
                               double *out_stream, double *normed,
                               int64_t rows, int64_t n,
                               double eps_post, double eps_pre, int stream_bf16)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *br = block_out + r * n;
        const double *rr = residual + r * n;
        double *sr = out_stream + r * n;
        double *nr = normed + r * n;

        /* post norm of the block output, then the residual add */
        double inv_post = row_inv_rms(br, n, eps_post);
        for (int64_t j = 0; j < n; ++j) {
            double s = br[j] * inv_post * gamma_post[j] + rr[j];
            if (stream_bf16)
                s = oracle_double_from_bf16(oracle_bf16_from_double(s));
            sr[j] = s;
        }

        /* pre norm of the stored stream */
        double inv_pre = row_inv_rms(sr, n, eps_pre);
        for (int64_t j = 0; j < n; ++j)
            nr[j] = sr[j] * inv_pre * gamma_pre[j];
    }
}

void oracle_add_rmsnorm(const double *a, const double *b, const double *gamma,
                        double *residual_out, double *normed,
                        int64_t rows, int64_t n, double eps, int sum_bf16)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *ar = a + r * n;
        const double *br = b + r * n;
        double *sr = residual_out + r * n;
        double *nr = normed + r * n;

        /* residual add; the stored sum is what the norm reads */
        for (int64_t j = 0; j < n; ++j) {
            double s = ar[j] + br[j];
            if (sum_bf16)
                s = oracle_double_from_bf16(oracle_bf16_from_double(s));
            sr[j] = s;
        }
        double inv_rms = row_inv_rms(sr, n, eps);
        for (int64_t j = 0; j < n; ++j)
            nr[j] = sr[j] * inv_rms * gamma[j];
    }
}

void oracle_rmsnorm_then_add_scale(const double *x, const double *gamma,
                                   const double *residual, double out_scale, double *out,
                                   int64_t rows, int64_t n, double eps)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * n;
        const double *rr = residual + r * n;
        double *outr = out + r * n;
        double inv_rms = row_inv_rms(xr, n, eps);
        for (int64_t j = 0; j < n; ++j)
            outr[j] = (xr[j] * inv_rms * gamma[j] + rr[j]) * out_scale;
    }
}

int oracle_q8_round(double qreal)
{
    double r = nearbyint(qreal);          /* default rounding: nearest, ties to even */
    if (r > 127.0)
        r = 127.0;
    if (r < -128.0)
        r = -128.0;
    return (int)r;
}

void oracle_rmsnorm_q8_1(const double *x, const double *gamma, int64_t rows, int64_t n,
                         double eps, double *d, double *qreal, int8_t *q)
{
    const int64_t blocks = n / 32;
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * n;
        double inv_rms = row_inv_rms(xr, n, eps);
        for (int64_t b = 0; b < blocks; ++b) {
            double normed[32];
            double amax = 0.0;
            for (int l = 0; l < 32; ++l) {
                int64_t j = b * 32 + l;
                normed[l] = xr[j] * gamma[j] * inv_rms;
                if (fabs(normed[l]) > amax)
                    amax = fabs(normed[l]);
            }
            double scale = amax / 127.0;
            d[r * blocks + b] = scale;
            for (int l = 0; l < 32; ++l) {
                int64_t j = r * n + b * 32 + l;
                qreal[j] = (scale == 0.0) ? 0.0 : normed[l] / scale;
                q[j] = (int8_t)oracle_q8_round(qreal[j]);
            }
        }
    }
}

/* value of the nearest T (binary16 or bf16) to v */
static double round_to_seam(double v, int seam_bf16)
{
    if (seam_bf16)
        return oracle_double_from_bf16(oracle_bf16_from_double(v));
    return oracle_double_from_f16(oracle_f16_from_double(v));
}

void oracle_rmsnorm_seam(const double *x, const double *gamma, double *u, double *y,
                         int64_t rows, int64_t n, double eps, int seam_bf16)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * n;
        double *ur = u + r * n;
        double *yr = y + r * n;
        double inv_rms = row_inv_rms(xr, n, eps);
        /* first operation: the weightless norm, published in T */
        for (int64_t j = 0; j < n; ++j)
            ur[j] = round_to_seam(xr[j] * inv_rms, seam_bf16);
        /* second operation: the weight multiply, rounded to T again */
        for (int64_t j = 0; j < n; ++j)
            yr[j] = round_to_seam(ur[j] * gamma[j], seam_bf16);
    }
}

/*
 * binary16: normal numbers (1 + f/1024) * 2^(e-15), e in 1..30; subnormals
 * f * 2^-24; e = 31 holds infinities and NaNs.  Same rounding rule as bf16.
 */
uint16_t oracle_f16_from_double(double v)
{
    if (isnan(v))
        return (uint16_t)0x7E00u;
    uint16_t sign = signbit(v) ? (uint16_t)0x8000u : (uint16_t)0;
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);
    int lead = e2 - 1;
    int quantum = (lead < -14) ? -24 : lead - 10;
    double scaled = ldexp(a, -quantum);
    double whole = floor(scaled);
    double frac = scaled - whole;
    uint64_t q = (uint64_t)whole;
    if (frac > 0.5 || (frac == 0.5 && (q & 1u)))
        q += 1;
    if (lead < -14)
        return (uint16_t)(sign | (uint16_t)q);     /* q == 1024 is the smallest normal */
    if (q == 2048) {
        q = 1024;
        lead += 1;
    }
    if (lead > 15)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(((lead + 15) << 10) | (int)(q - 1024)));
}

double oracle_double_from_f16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int field = (bits >> 10) & 0x1F;
    int frac = bits & 0x3FF;
    double v;
    if (field == 0x1F)
        v = frac ? NAN : INFINITY;
    else if (field == 0)
        v = ldexp((double)frac, -24);
    else
        v = ldexp((double)(1024 + frac), field - 15 - 10);
    return sign ? -v : v;
}

/*
 * bf16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.  Normal
 * numbers are (1 + f/128) * 2^(e-127) for e in 1..254; e = 0 holds the
 * subnormals f * 2^-133; e = 255 holds infinities (f = 0) and NaNs.
 * Rounding: pick the representable neighbour nearest to v; on an exact tie,
 * the one whose last significand bit is 0.
 */
uint16_t oracle_bf16_from_double(double v)
{
    if (isnan(v))
        return (uint16_t)0x7FC0u;
    uint16_t sign = signbit(v) ? (uint16_t)0x8000u : (uint16_t)0;
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;

    int e2;
    (void)frexp(a, &e2);          /* a = m * 2^e2 with m in [0.5, 1) */
    int lead = e2 - 1;            /* a lies in [2^lead, 2^(lead+1)) */
    /* exponent of one unit in the last place of the target format */
    int quantum = (lead < -126) ? -133 : lead - 7;

    double scaled = ldexp(a, -quantum);   /* exact: a power-of-two scale */
    double whole = floor(scaled);
    double frac = scaled - whole;         /* exact */
    uint64_t q = (uint64_t)whole;
    if (frac > 0.5 || (frac == 0.5 && (q & 1u)))
        q += 1;

    if (lead < -126) {
        /* subnormal range; q == 128 is the smallest normal, whose encoding
         * (exponent field 1, fraction 0) is again the integer 128 */
        return (uint16_t)(sign | (uint16_t)q);
    }
    if (q == 256) {               /* rounding carried into the next binade */
        q = 128;
        lead += 1;
    }
    if (lead > 127)
        return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)(((lead + 127) << 7) | (int)(q - 128)));
}

double oracle_double_from_bf16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int field = (bits >> 7) & 0xFF;
    int frac = bits & 0x7F;
    double v;
    if (field == 0xFF)
        v = frac ? NAN : INFINITY;
    else if (field == 0)
        v = ldexp((double)frac, -133);
    else
        v = ldexp((double)(128 + frac), field - 127 - 7);
    return sign ? -v : v;
}

void oracle_bf16_round_array(const double *v, uint16_t *bits, int64_t count)
{
    for (int64_t i = 0; i < count; ++i)
        bits[i] = oracle_bf16_from_double(v[i]);
}

void oracle_bf16_widen_array(const uint16_t *bits, double *v, int64_t count)
{
    for (int64_t i = 0; i < count; ++i)
        v[i] = oracle_double_from_bf16(bits[i]);
}
