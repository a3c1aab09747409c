/*
 * Row-normalization oracle: plain, slow, fp64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library under row_normalization_inner_gb300/csrc.
 *
 * Sources for what is computed:
 *   - "optimize inner persistent scheduler for static fusion" (NVIDIA/Fuser
 *     PR #5281), changes walkthrough, test_rmsnorm_add_fwd.py entry: the
 *     fused residual-add + RMSNorm forward with in-place update semantics.
 *   - "TMA inner persistent scheduler" (NVIDIA/Fuser PR #5587), description:
 *     RMS norm and layer norm (forward) implementations.
 *   - "Llu/ln bwd" (NVIDIA/Fuser PR #207), title and the design discussion:
 *     layer norm backward as a combined per-row (inner) and across-rows
 *     (outer) reduction.
 * The pages name these operations but print no formulas; the formulas below
 * are the textbook definitions of RMSNorm and LayerNorm, with eps added to
 * the mean square / biased variance inside the square root.
 *
 * Every function here takes and returns double arrays, row-major
 * [rows, hidden], and loops in the plainest order.  Conversion between bf16
 * bit patterns and double is done by the two helpers at the top.  Each loop
 * is a direct transcription of the definition; there is no blocking, fusion
 * or reordering.
 *
 * Pins (tests/test_oracle.py): bf16 conversion against torch's own
 * conversions; RMSNorm against the closed form mean(y^2) = ms/(ms+eps) (w=1),
 * scale invariance, a hand-computed H=4 case and torch.nn.functional.rms_norm
 * in fp64; LayerNorm forward against mean(y)=0, var(y)=var/(var+eps), shift
 * invariance, constant rows and torch.nn.functional.layer_norm in fp64;
 * LayerNorm backward against central finite differences of sum(dy*LN(x)),
 * the per-row invariants sum(dx)=0 and sum(dx*xhat)=0 (gamma=1), and torch
 * autograd in fp64.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

/* ---- bf16 <-> double --------------------------------------------------- */

/* A bf16 value is the upper half of an IEEE binary32 bit pattern, so
 * widening is exact: shift the 16 bits into the high half of a float. */
double or_bf16_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even, in ONE rounding
 * (no detour through binary32, which could round twice).
 *
 * bf16 keeps 8 significant bits (1 implicit + 7 stored) and binary32's
 * exponent range: normals down to 2^-126, subnormals spaced 2^-133, largest
 * finite (2 - 2^-7) * 2^127.  For |d| in [2^e, 2^(e+1)) the spacing of bf16
 * values is q = 2^(e-7), but never below 2^-133.  d/q is then exact (q is a
 * power of two), nearbyint() rounds it to an integer with ties to even under
 * the default rounding mode, and the product is the rounded value, which
 * binary32 holds exactly, so its top 16 bits are the answer. */
uint16_t or_double_to_bf16(double d) {
    uint32_t bits;
    float f;
    if (isnan(d)) return (uint16_t)0x7FC0u;
    if (d == 0.0) {
        f = (float)d; /* keeps the sign of zero */
        memcpy(&bits, &f, sizeof bits);
        return (uint16_t)(bits >> 16);
    }
    if (isinf(d)) return d > 0 ? (uint16_t)0x7F80u : (uint16_t)0xFF80u;
    int e2;
    frexp(d, &e2);              /* |d| = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;             /* |d| in [2^e, 2^(e+1)) */
    int qexp = e - 7;
    if (qexp < -133) qexp = -133;
    double q = ldexp(1.0, qexp);
    double r = nearbyint(d / q) * q;
    /* Beyond the largest finite bf16 the rounded magnitude is 2^128. */
    if (fabs(r) >= ldexp(1.0, 128)) return d > 0 ? (uint16_t)0x7F80u : (uint16_t)0xFF80u;
    f = (float)r;               /* exact */
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(bits >> 16);
}

void or_bf16_to_double_array(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_to_double(h[i]);
}

void or_double_to_bf16_array(const double* d, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_double_to_bf16(d[i]);
}

/* ---- RMSNorm forward ------------------------------------------------------
 * y[r][j] = x[r][j] / sqrt(ms_r + eps) * w[j],  ms_r = (1/H) sum_j x[r][j]^2.
 * rstd_out (optional) receives 1/sqrt(ms_r + eps) per row. */
void or_rmsnorm_fwd(const double* x, const double* w, int64_t rows, int64_t hidden,
                    double eps, double* y, double* rstd_out) {
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * hidden;
        double ss = 0.0;
        for (int64_t j = 0; j < hidden; ++j) ss += xr[j] * xr[j];
        double ms = ss / (double)hidden;
        double inv = 1.0 / sqrt(ms + eps);
        for (int64_t j = 0; j < hidden; ++j) y[r * hidden + j] = xr[j] * inv * w[j];
        if (rstd_out) rstd_out[r] = inv;
    }
}

/* ---- fused residual add + RMSNorm forward, in place ------------------------
 * residual <- residual + x ;  x <- RMSNorm(residual) * w.
 * The sum s = x + residual is exact in double for bf16 inputs.  s_out gets
 * s (the caller rounds it to bf16 for the stored residual).  y gets the
 * normalized row.
 *
 * normalize_rounded: 0 normalizes the exact sum s (the reading used by the
 * parity tests: the kernel holds the unrounded sum anyway); 1 normalizes
 * bf16(s), the literal "residual after the in-place update" reading.  The
 * two differ by at most half a bf16 ulp relative before the final rounding. */
void or_fused_add_rmsnorm(const double* x, const double* residual, const double* w,
                          int64_t rows, int64_t hidden, double eps, int normalize_rounded,
                          double* s_out, double* y, double* rstd_out) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < hidden; ++j) {
            double s = x[r * hidden + j] + residual[r * hidden + j];
            if (normalize_rounded) s = or_bf16_to_double(or_double_to_bf16(s));
            s_out[r * hidden + j] = s;
        }
    }
    or_rmsnorm_fwd(s_out, w, rows, hidden, eps, y, rstd_out);
}

/* ---- LayerNorm forward -----------------------------------------------------
 * mean_r = (1/H) sum_j x ; var_r = (1/H) sum_j (x - mean_r)^2 (biased) ;
 * rstd_r = 1/sqrt(var_r + eps) ; y = (x - mean_r) * rstd_r * gamma + beta. */
void or_layernorm_fwd(const double* x, const double* gamma, const double* beta,
                      int64_t rows, int64_t hidden, double eps,
                      double* y, double* mean_out, double* rstd_out) {
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * hidden;
        double sum = 0.0;
        for (int64_t j = 0; j < hidden; ++j) sum += xr[j];
        double mean = sum / (double)hidden;
        double sq = 0.0;
        for (int64_t j = 0; j < hidden; ++j) sq += (xr[j] - mean) * (xr[j] - mean);
        double var = sq / (double)hidden;
        double rstd = 1.0 / sqrt(var + eps);
        for (int64_t j = 0; j < hidden; ++j)
            y[r * hidden + j] = (xr[j] - mean) * rstd * gamma[j] + beta[j];
        if (mean_out) mean_out[r] = mean;
        if (rstd_out) rstd_out[r] = rstd;
    }
}

/* ---- LayerNorm backward ----------------------------------------------------
 * With y = xhat * gamma + beta, xhat = (x - mean) * rstd and the saved
 * mean/rstd treated as functions of x, the gradient of L = sum dy * y is
 *   per row (inner reduction over j):
 *     g_j   = dy_j * gamma_j
 *     dx_j  = rstd * ( g_j - (1/H) sum_k g_k - xhat_j * (1/H) sum_k g_k * xhat_k )
 *   per column (outer reduction over rows r):
 *     dgamma_j = sum_r dy[r][j] * xhat[r][j]
 *     dbeta_j  = sum_r dy[r][j]
 * mean and rstd are inputs (the values saved by the forward). */
void or_layernorm_bwd(const double* dy, const double* x, const double* mean,
                      const double* rstd, const double* gamma,
                      int64_t rows, int64_t hidden,
                      double* dx, double* dgamma, double* dbeta) {
    for (int64_t j = 0; j < hidden; ++j) { dgamma[j] = 0.0; dbeta[j] = 0.0; }
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * hidden;
        const double* dyr = dy + r * hidden;
        double sum_g = 0.0, sum_gx = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            double xhat = (xr[j] - mean[r]) * rstd[r];
            double g = dyr[j] * gamma[j];
            sum_g += g;
            sum_gx += g * xhat;
        }
        double mean_g = sum_g / (double)hidden;
        double mean_gx = sum_gx / (double)hidden;
        for (int64_t j = 0; j < hidden; ++j) {
            double xhat = (xr[j] - mean[r]) * rstd[r];
            double g = dyr[j] * gamma[j];
            dx[r * hidden + j] = rstd[r] * (g - mean_g - xhat * mean_gx);
        }
    }
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < hidden; ++j) {
            double xhat = (x[r * hidden + j] - mean[r]) * rstd[r];
            dgamma[j] += dy[r * hidden + j] * xhat;
            dbeta[j] += dy[r * hidden + j];
        }
    }
}

/* ---- RMSNorm backward ------------------------------------------------------
 * With y = xhat * w, xhat = x * rstd and rstd = (mean(x^2) + eps)^(-1/2)
 * treated as a function of x, the gradient of L = sum dy * y is
 *   per row:     g_j  = dy_j * w_j
 *                dx_j = rstd * ( g_j - xhat_j * (1/H) sum_k g_k * xhat_k )
 *   per column:  dw_j = sum_r dy[r][j] * xhat[r][j]
 * rstd is an input (the value saved by the forward). */
void or_rmsnorm_bwd(const double* dy, const double* x, const double* rstd, const double* w,
                    int64_t rows, int64_t hidden, double* dx, double* dw) {
    for (int64_t j = 0; j < hidden; ++j) dw[j] = 0.0;
    for (int64_t r = 0; r < rows; ++r) {
        double sum_gx = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            double xhat = x[r * hidden + j] * rstd[r];
            sum_gx += dy[r * hidden + j] * w[j] * xhat;
        }
        double mean_gx = sum_gx / (double)hidden;
        for (int64_t j = 0; j < hidden; ++j) {
            double xhat = x[r * hidden + j] * rstd[r];
            double g = dy[r * hidden + j] * w[j];
            dx[r * hidden + j] = rstd[r] * (g - xhat * mean_gx);
        }
    }
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < hidden; ++j)
            dw[j] += dy[r * hidden + j] * x[r * hidden + j] * rstd[r];
}

/* ---- fused add + RMSNorm backward ------------------------------------------
 * The forward leaves s = x + residual in the residual buffer and overwrites x
 * with y = s * rstd(s) * w, so the backward sees s (as saved) and two
 * incoming gradients: dy for y and dres for the residual stream s.  Both
 * inputs x and residual receive the same gradient
 *   ds = rmsnorm_bwd(dy, s, w) + dres,   dw = sum_r dy * s * rstd(s),
 * with rstd(s) = 1 / sqrt(mean(s^2) + eps) recomputed from s.  dres may be
 * NULL (no residual-stream gradient). */
void or_fused_add_rmsnorm_bwd(const double* dy, const double* dres, const double* s,
                              const double* w, int64_t rows, int64_t hidden, double eps,
                              double* ds, double* dw) {
    double* rstd = (double*)malloc((size_t)(rows > 0 ? rows : 1) * sizeof(double));
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t j = 0; j < hidden; ++j) ss += s[r * hidden + j] * s[r * hidden + j];
        rstd[r] = 1.0 / sqrt(ss / (double)hidden + eps);
    }
    or_rmsnorm_bwd(dy, s, rstd, w, rows, hidden, ds, dw);
    if (dres)
        for (int64_t i = 0; i < rows * hidden; ++i) ds[i] += dres[i];
    free(rstd);
}

/* ---- outer normalization (per column, over the rows) -----------------------
 * "Llu/ln bwd" lists block- and grid-parallel outer normalization among the
 * normalization variants: the statistics run across the rows, one set per
 * column (batch normalization of a [rows, hidden] matrix, training mode):
 *   mean_j = (1/R) sum_r x[r][j] ; var_j = (1/R) sum_r (x[r][j] - mean_j)^2 (biased)
 *   rstd_j = 1/sqrt(var_j + eps) ; y[r][j] = (x[r][j] - mean_j) * rstd_j * gamma[j] + beta[j] */
void or_outer_norm_fwd(const double* x, const double* gamma, const double* beta,
                       int64_t rows, int64_t hidden, double eps,
                       double* y, double* mean_out, double* rstd_out) {
    for (int64_t j = 0; j < hidden; ++j) {
        double sum = 0.0;
        for (int64_t r = 0; r < rows; ++r) sum += x[r * hidden + j];
        double mean = sum / (double)rows;
        double sq = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
            double d = x[r * hidden + j] - mean;
            sq += d * d;
        }
        double var = sq / (double)rows;
        double rstd = 1.0 / sqrt(var + eps);
        for (int64_t r = 0; r < rows; ++r)
            y[r * hidden + j] = (x[r * hidden + j] - mean) * rstd * gamma[j] + beta[j];
        if (mean_out) mean_out[j] = mean;
        if (rstd_out) rstd_out[j] = rstd;
    }
}

/* Gradient of L = sum dy * y for the outer normalization above, with the
 * saved per-column mean/rstd treated as functions of x:
 *   xhat = (x - mean_j) * rstd_j ; g = dy * gamma[j]
 *   dx[r][j] = rstd_j * ( g - (1/R) sum_s g[s][j] - xhat * (1/R) sum_s g[s][j] * xhat[s][j] )
 *   dgamma[j] = sum_r dy[r][j] * xhat[r][j] ; dbeta[j] = sum_r dy[r][j] */
void or_outer_norm_bwd(const double* dy, const double* x, const double* mean, const double* rstd,
                       const double* gamma, int64_t rows, int64_t hidden,
                       double* dx, double* dgamma, double* dbeta) {
    for (int64_t j = 0; j < hidden; ++j) {
        double sum_g = 0.0, sum_gx = 0.0, sum_dy = 0.0, sum_dyx = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
            double xhat = (x[r * hidden + j] - mean[j]) * rstd[j];
            double g = dy[r * hidden + j] * gamma[j];
            sum_g += g;
            sum_gx += g * xhat;
            sum_dy += dy[r * hidden + j];
            sum_dyx += dy[r * hidden + j] * xhat;
        }
        double mean_g = sum_g / (double)rows;
        double mean_gx = sum_gx / (double)rows;
        for (int64_t r = 0; r < rows; ++r) {
            double xhat = (x[r * hidden + j] - mean[j]) * rstd[j];
            double g = dy[r * hidden + j] * gamma[j];
            dx[r * hidden + j] = rstd[j] * (g - mean_g - xhat * mean_gx);
        }
        dgamma[j] = sum_dyx;
        dbeta[j] = sum_dy;
    }
}
