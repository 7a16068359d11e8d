/*
 * norm_oracle.c -- plain FP64 CPU oracle for row-wise RMSNorm, LayerNorm and
 * FusedAddRMSNorm, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg load it.  It shares no code, header or constant with the CUDA
 * kernels.
 *
 * Conventions
 *   - Every tensor is a dense row-major array of doubles.  Row i of an M x N
 *     matrix is a[i*N .. i*N+N-1].  Inputs are the exact values of the
 *     (already rounded) tensors the kernels see.
 *   - All arithmetic is FP64, in the order the formulas are written, one row
 *     after another.  Nothing is blocked, fused or reordered.
 *   - The per-column scale is W'_j = w_j + offset, formed in FP64 from the
 *     stored weight, never from a pre-rounded (w + offset).  This is the fix
 *     described on "fix(cutedsl): fuse Gemma RMSNorm weight offset in FP32",
 *     Summary.
 *   - The normalisation constant is rstd = 1 / sqrt(mean + eps) with eps
 *     inside the square root (the pages print no formula; this is the
 *     standard reading).  LayerNorm uses the biased (1/N) variance.
 *   - The backward entry points take the statistics the forward saved (rstd,
 *     and the mean for LayerNorm) as optional inputs; given NULL they
 *     recompute them from their input rows in FP64.
 *   - Rounding of an FP64 result to bf16 / fp16 / fp32 is done once, directly
 *     from FP64, round-to-nearest, ties-to-even (oracle_round_*).
 *
 * Optional outputs named *_scale hold, per element, the magnitude of the
 * terms whose sum forms that output, where a row constant that is itself a
 * sum (c = mean of g*xhat) contributes the mean of its terms' magnitudes
 * (for an RMSNorm input gradient: rstd*(|g_j| + |xhat_j| * mean|g xhat|)).
 * The tests use them to bound FP32 cancellation error; they play no part in
 * the outputs themselves.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* RMSNorm                                                                   */
/* ------------------------------------------------------------------------ */

/* Root mean square of one row, as 1/sqrt(mean(x^2) + eps). */
static double row_rstd_rms(const double *xr, int64_t N, double eps)
{
    double ss = 0.0;
    for (int64_t j = 0; j < N; ++j)
        ss += xr[j] * xr[j];
    double ms = ss / (double)N;
    return 1.0 / sqrt(ms + eps);
}

/*
 * RMSNorm forward: y_ij = x_ij * rstd_i * (w_j + offset).
 * The operation whose backward is specialised on
 * "perf(norm): skip dW/dB calculation when parameters are frozen", Key Changes
 * (rms_norm), with the weight offset of
 * "fix(cutedsl): fuse Gemma RMSNorm weight offset in FP32", Summary.
 * rstd (length M) is optional.
 */
void oracle_rms_fwd(int64_t M, int64_t N, const double *x, const double *w,
                    double offset, double eps, double *y, double *rstd)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *xr = x + i * N;
        double r = row_rstd_rms(xr, N, eps);
        for (int64_t j = 0; j < N; ++j)
            y[i * N + j] = xr[j] * r * (w[j] + offset);
        if (rstd)
            rstd[i] = r;
    }
}

/*
 * RMSNorm backward, the gradient of the forward above:
 *   xhat_j = x_j * rstd,  g_j = dy_j * (w_j + offset),
 *   c      = (1/N) * sum_j g_j * xhat_j,
 *   dx_j   = rstd * (g_j - xhat_j * c),
 *   dw_j   = sum over rows of dy_j * xhat_j          (only if dw != NULL).
 * The offset is a constant, so dw is the same whether the learned parameter
 * is w or w + offset ("fix(cutedsl): ...", PyTorch accuracy comparison: dW is
 * unchanged).  A NULL dw is the frozen-weight case of
 * "perf(norm): skip dW/dB calculation when parameters are frozen", Motivation.
 * rstd_in: the statistic saved by the forward (length M), or NULL to
 * recompute it from x.  The formula is applied with whichever rstd is used.
 * dx_scale_j = rstd*(|g_j| + |xhat_j| * (1/N) sum_k |g_k xhat_k|): the size of
 * the terms dx_j is formed from, with c replaced by the size of its terms.
 */
void oracle_rms_bwd(int64_t M, int64_t N, const double *x, const double *dy,
                    const double *w, double offset, double eps, double *dx,
                    double *dw, double *dx_scale, const double *rstd_in)
{
    if (dw)
        for (int64_t j = 0; j < N; ++j)
            dw[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        const double *xr = x + i * N;
        const double *dyr = dy + i * N;
        double r = rstd_in ? rstd_in[i] : row_rstd_rms(xr, N, eps);
        double sgx = 0.0, sgx_abs = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double gx = dyr[j] * (w[j] + offset) * (xr[j] * r);
            sgx += gx;
            sgx_abs += fabs(gx);
        }
        double c = sgx / (double)N;
        double c_abs = sgx_abs / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double xhat = xr[j] * r;
            double g = dyr[j] * (w[j] + offset);
            dx[i * N + j] = r * (g - xhat * c);
            if (dx_scale)
                dx_scale[i * N + j] = r * (fabs(g) + fabs(xhat) * c_abs);
            if (dw)
                dw[j] += dyr[j] * xhat;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* LayerNorm                                                                 */
/* ------------------------------------------------------------------------ */

static void row_stats_ln(const double *xr, int64_t N, double eps,
                         double *mean_out, double *rstd_out)
{
    double s = 0.0;
    for (int64_t j = 0; j < N; ++j)
        s += xr[j];
    double mu = s / (double)N;
    double sq = 0.0;
    for (int64_t j = 0; j < N; ++j)
        sq += (xr[j] - mu) * (xr[j] - mu);
    double var = sq / (double)N;
    *mean_out = mu;
    *rstd_out = 1.0 / sqrt(var + eps);
}

/*
 * LayerNorm forward: y_ij = (x_ij - mean_i) * rstd_i * (w_j + offset) + b_j,
 * biased variance.  b may be NULL (no bias).  mean, rstd, y_scale optional.
 * "perf(norm): skip dW/dB calculation when parameters are frozen",
 * Key Changes (layer_norm).
 */
void oracle_ln_fwd(int64_t M, int64_t N, const double *x, const double *w,
                   const double *b, double offset, double eps, double *y,
                   double *mean, double *rstd, double *y_scale)
{
    for (int64_t i = 0; i < M; ++i) {
        const double *xr = x + i * N;
        double mu, r;
        row_stats_ln(xr, N, eps, &mu, &r);
        for (int64_t j = 0; j < N; ++j) {
            double bj = b ? b[j] : 0.0;
            y[i * N + j] = (xr[j] - mu) * r * (w[j] + offset) + bj;
            if (y_scale)
                y_scale[i * N + j] =
                    (fabs(xr[j]) + fabs(mu)) * r * fabs(w[j] + offset) + fabs(bj);
        }
        if (mean)
            mean[i] = mu;
        if (rstd)
            rstd[i] = r;
    }
}

/*
 * LayerNorm backward:
 *   xhat_j = (x_j - mean) * rstd,  g_j = dy_j * (w_j + offset),
 *   dx_j   = rstd * (g_j - (1/N) sum_k g_k - xhat_j * (1/N) sum_k g_k xhat_k),
 *   dw_j   = sum over rows of dy_j * xhat_j   (if dw != NULL),
 *   db_j   = sum over rows of dy_j            (if db != NULL).
 * dw and db are independent, as on "perf(norm): skip dW/dB calculation when
 * parameters are frozen", Key Changes (layer_norm).
 * mean_in / rstd_in: the statistics saved by the forward, or both NULL to
 * recompute them from x.
 */
void oracle_ln_bwd(int64_t M, int64_t N, const double *x, const double *dy,
                   const double *w, double offset, double eps, double *dx,
                   double *dw, double *db, double *dx_scale,
                   const double *mean_in, const double *rstd_in)
{
    if (dw)
        for (int64_t j = 0; j < N; ++j)
            dw[j] = 0.0;
    if (db)
        for (int64_t j = 0; j < N; ++j)
            db[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        const double *xr = x + i * N;
        const double *dyr = dy + i * N;
        double mu, r;
        if (mean_in && rstd_in) {
            mu = mean_in[i];
            r = rstd_in[i];
        } else {
            row_stats_ln(xr, N, eps, &mu, &r);
        }
        double sg = 0.0, sgx = 0.0, sg_abs = 0.0, sgx_abs = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double g = dyr[j] * (w[j] + offset);
            double gx = g * ((xr[j] - mu) * r);
            sg += g;
            sgx += gx;
            sg_abs += fabs(g);
            sgx_abs += fabs(gx);
        }
        double mg = sg / (double)N;
        double mgx = sgx / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double xhat = (xr[j] - mu) * r;
            double g = dyr[j] * (w[j] + offset);
            dx[i * N + j] = r * (g - mg - xhat * mgx);
            if (dx_scale)
                dx_scale[i * N + j] = r * (fabs(g) + sg_abs / (double)N
                                           + fabs(xhat) * sgx_abs / (double)N);
            if (dw)
                dw[j] += dyr[j] * xhat;
            if (db)
                db[j] += dyr[j];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* FusedAddRMSNorm                                                           */
/* ------------------------------------------------------------------------ */

/*
 * FusedAddRMSNorm forward: h = x + residual (exact in FP64), y = RMSNorm(h)
 * with scale (w + offset).  Outputs y, h (the residual stream passed on) and
 * optionally rstd.  "perf(norm): skip dW/dB ...", Key Changes
 * (fused_add_rms_norm); "fix(cutedsl): ...", Summary.
 */
void oracle_fused_add_rms_fwd(int64_t M, int64_t N, const double *x,
                              const double *residual, const double *w,
                              double offset, double eps, double *y, double *h,
                              double *rstd)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            h[i * N + j] = x[i * N + j] + residual[i * N + j];
    oracle_rms_fwd(M, N, h, w, offset, eps, y, rstd);
}

/*
 * FusedAddRMSNorm backward from the forward's saved tensors: the residual
 * stream h as the kernel stores it (rounded to the activation type --
 * "fix(cutedsl): ...", PyTorch accuracy comparison: the backward uses a
 * rounded saved residual) and the forward's rstd of the unrounded sum
 * (rstd_in; NULL recomputes it from h).  The RMSNorm input-gradient formula
 * is applied to those saved values and the gradient dh_out arriving on the
 * residual-stream output (NULL = zero) is added.  The result is both dx and
 * dresidual, since h = x + residual.
 */
void oracle_fused_add_rms_bwd(int64_t M, int64_t N, const double *h,
                              const double *dy, const double *dh_out,
                              const double *w, double offset, double eps,
                              double *dx, double *dw, double *dx_scale,
                              const double *rstd_in)
{
    oracle_rms_bwd(M, N, h, dy, w, offset, eps, dx, dw, dx_scale, rstd_in);
    if (dh_out) {
        for (int64_t i = 0; i < M * N; ++i) {
            dx[i] = dx[i] + dh_out[i];
            if (dx_scale)
                dx_scale[i] = dx_scale[i] + fabs(dh_out[i]);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Rounding FP64 -> storage types, round to nearest, ties to even            */
/* ------------------------------------------------------------------------ */

/*
 * Round |a| (finite, > 0) to a binary floating-point grid with `mbits`
 * explicit mantissa bits and minimum normal exponent `emin`: the spacing in
 * [2^E, 2^(E+1)) is 2^(E - mbits), and below 2^emin it stays 2^(emin - mbits)
 * (subnormals).  a / q is exact because q is a power of two, and nearbyint
 * rounds to the nearest integer with ties to even (default rounding mode).
 */
static double round_grid(double a, int mbits, int emin)
{
    int k;
    (void)frexp(a, &k);            /* a = m * 2^k, m in [0.5, 1) */
    int E = k - 1;                 /* a in [2^E, 2^(E+1)) */
    if (E < emin)
        E = emin;
    double q = ldexp(1.0, E - mbits);
    double n = nearbyint(a / q);
    return n * q;
}

/* bfloat16: 8 exponent bits (bias 127), 7 explicit mantissa bits. */
uint16_t oracle_round_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    double r = round_grid(a, 7, -126);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    if (r == 0.0)
        return sign;
    /* r is exactly representable in bfloat16, hence in float: take the top
       half of its binary32 encoding. */
    float f = (float)r;
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return sign | (uint16_t)(bits >> 16);
}

/* IEEE binary16: 5 exponent bits (bias 15), 10 explicit mantissa bits. */
uint16_t oracle_round_f16(double v)
{
    if (isnan(v))
        return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7C00;
    double r = round_grid(a, 10, -14);
    if (r >= 65536.0)
        return sign | 0x7C00;
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -14)) {     /* subnormal: r = m * 2^-24, m < 1024 */
        uint16_t m = (uint16_t)(r / ldexp(1.0, -24));
        return sign | m;
    }
    int k;
    double m = frexp(r, &k);       /* r = m * 2^k, m in [0.5, 1) */
    int E = k - 1;
    uint16_t frac = (uint16_t)((m * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | frac;
}

/* IEEE binary32: the C conversion rounds to nearest, ties to even. */
float oracle_round_f32(double v)
{
    return (float)v;
}

/* Array forms: dtype 0 = float32 (out is float*), 1 = float16, 2 = bfloat16
   (out is uint16_t* holding the bit patterns). */
void oracle_round_array(const double *in, int64_t n, int dtype, void *out)
{
    for (int64_t i = 0; i < n; ++i) {
        if (dtype == 0)
            ((float *)out)[i] = oracle_round_f32(in[i]);
        else if (dtype == 1)
            ((uint16_t *)out)[i] = oracle_round_f16(in[i]);
        else
            ((uint16_t *)out)[i] = oracle_round_bf16(in[i]);
    }
}
