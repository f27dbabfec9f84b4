/*
 * norm_oracle.c -- float64 CPU oracle for the LayerNorm / RMSNorm forward and
 * backward passes.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library.  The CUDA library shares no code,
 * header, table or helper with it.
 *
 * Every function is the textbook definition written out row by row in double
 * precision, with plain left-to-right sums and no blocking, fusion or
 * reordering.  Inputs are the storage values already widened to double.
 *
 * Sources (pages about the method):
 *   [NB]  "Norm backward in Triton -- the dγ/dβ reduction", section
 *         "The gradients": mu = mean(x), sigma = sqrt(var(x) + eps),
 *         xhat = (x - mu) / sigma, y = gamma * xhat + beta; dyhat = dy * gamma,
 *         dx = (1/sigma) [dyhat - mean(dyhat) - xhat * mean(dyhat * xhat)],
 *         dgamma = sum over rows of dy * xhat, dbeta = sum over rows of dy;
 *         RMSNorm: xhat = x / sigma, sigma = sqrt(mean(x^2) + eps), and dx
 *         loses the mean(dyhat) term.
 *   [NA]  "Norm & activation backward", section "LayerNorm backward, derived"
 *         (same formulas) and section "Half one" (the backward takes the saved
 *         per-row statistic instead of a stored xhat).
 *   [LN5] "05: Layer norm", kernel ln_fwd: the variance is the biased one,
 *         sum((x - mu)^2) / N, computed after the mean (two passes), and
 *         eps is added under the square root.
 *
 * Readings where the pages leave a choice open:
 *   - variance divides by N (biased), as ln_fwd does;
 *   - eps is added to var (LayerNorm) or mean(x^2) (RMSNorm) under the root;
 *   - RMSNorm has no beta and no dbeta;
 *   - the backward uses the saved mean / rstd it is given (rstd = 1/sigma);
 *   - M = 0 gives dgamma = dbeta = 0.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fused multiply-add, so
 * x86-64 and aarch64 hosts give identical results).
 */
#include <math.h>
#include <stdint.h>

/* LayerNorm forward, [NB] "The gradients" (forward line) and [LN5] ln_fwd. */
void oracle_ln_fwd(int64_t M, int64_t N, const double *x, const double *gamma,
                   const double *beta, double eps, double *y, double *mean,
                   double *rstd)
{
    for (int64_t r = 0; r < M; ++r) {
        const double *xr = x + r * N;
        double sum = 0.0;
        for (int64_t j = 0; j < N; ++j)
            sum += xr[j];
        const double mu = sum / (double)N;
        double sq = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double d = xr[j] - mu;
            sq += d * d;
        }
        const double var = sq / (double)N;
        const double rs = 1.0 / sqrt(var + eps);
        mean[r] = mu;
        rstd[r] = rs;
        for (int64_t j = 0; j < N; ++j) {
            const double xhat = (xr[j] - mu) * rs;
            y[r * N + j] = gamma[j] * xhat + beta[j];
        }
    }
}

/* RMSNorm forward, [NB] "The gradients" (RMSNorm paragraph). */
void oracle_rms_fwd(int64_t M, int64_t N, const double *x, const double *gamma,
                    double eps, double *y, double *rstd)
{
    for (int64_t r = 0; r < M; ++r) {
        const double *xr = x + r * N;
        double sq = 0.0;
        for (int64_t j = 0; j < N; ++j)
            sq += xr[j] * xr[j];
        const double ms = sq / (double)N;
        const double rs = 1.0 / sqrt(ms + eps);
        rstd[r] = rs;
        for (int64_t j = 0; j < N; ++j) {
            const double xhat = xr[j] * rs;
            y[r * N + j] = gamma[j] * xhat;
        }
    }
}

/*
 * LayerNorm backward, [NB] "The gradients" (the dx, dgamma, dbeta lines) and
 * [NA] "LayerNorm backward, derived".  xhat is recomputed from the saved
 * mean and rstd ([NA] "Half one").
 */
void oracle_ln_bwd(int64_t M, int64_t N, const double *dy, const double *x,
                   const double *gamma, const double *mean, const double *rstd,
                   double *dx, double *dgamma, double *dbeta)
{
    for (int64_t j = 0; j < N; ++j) {
        dgamma[j] = 0.0;
        dbeta[j] = 0.0;
    }
    for (int64_t r = 0; r < M; ++r) {
        const double *xr = x + r * N;
        const double *dyr = dy + r * N;
        const double mu = mean[r];
        const double rs = rstd[r];
        /* the two in-row reductions: mean(dyhat) and mean(dyhat * xhat) */
        double s1 = 0.0, s2 = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double xhat = (xr[j] - mu) * rs;
            const double dyhat = dyr[j] * gamma[j];
            s1 += dyhat;
            s2 += dyhat * xhat;
        }
        const double mean_dyhat = s1 / (double)N;
        const double mean_dyhat_xhat = s2 / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            const double xhat = (xr[j] - mu) * rs;
            const double dyhat = dyr[j] * gamma[j];
            dx[r * N + j] = rs * (dyhat - mean_dyhat - xhat * mean_dyhat_xhat);
            /* the cross-row, per-feature sums */
            dgamma[j] += dyr[j] * xhat;
            dbeta[j] += dyr[j];
        }
    }
}

/* RMSNorm backward: LayerNorm's with no mean and no mean(dyhat) term, no dbeta. */
void oracle_rms_bwd(int64_t M, int64_t N, const double *dy, const double *x,
                    const double *gamma, const double *rstd, double *dx,
                    double *dgamma)
{
    for (int64_t j = 0; j < N; ++j)
        dgamma[j] = 0.0;
    for (int64_t r = 0; r < M; ++r) {
        const double *xr = x + r * N;
        const double *dyr = dy + r * N;
        const double rs = rstd[r];
        double s2 = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double xhat = xr[j] * rs;
            const double dyhat = dyr[j] * gamma[j];
            s2 += dyhat * xhat;
        }
        const double mean_dyhat_xhat = s2 / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            const double xhat = xr[j] * rs;
            const double dyhat = dyr[j] * gamma[j];
            dx[r * N + j] = rs * (dyhat - xhat * mean_dyhat_xhat);
            dgamma[j] += dyr[j] * xhat;
        }
    }
}

/*
 * Activation backward, "Norm backward in Triton -- the dγ/dβ reduction",
 * section "Activation backward -- fuse it into the epilogue" (and "Norm &
 * activation backward", same section): dx = dy * f'(preact), the derivative
 * recomputed from the saved pre-activation.
 *   SiLU: f(x) = x * sigma(x), f'(x) = sigma(x) * (1 + x * (1 - sigma(x))).
 *   GELU (the pages name it without a formula; the exact erf form is taken):
 *   f(x) = x * Phi(x), f'(x) = Phi(x) + x * phi(x), Phi the standard normal
 *   distribution function, phi its density.  Phi(x) is evaluated as
 *   erfc(-x / sqrt 2) / 2, its definition through the complementary error
 *   function: the form (1 + erf(x / sqrt 2)) / 2 cancels to no correct digit
 *   in double below x = -8, where Phi is still far from negligible next to
 *   x * phi(x).
 */
void oracle_silu_bwd(int64_t n, const double *dy, const double *preact, double *dx)
{
    for (int64_t i = 0; i < n; ++i) {
        const double x = preact[i];
        const double s = 1.0 / (1.0 + exp(-x));
        dx[i] = dy[i] * (s * (1.0 + x * (1.0 - s)));
    }
}

void oracle_gelu_bwd(int64_t n, const double *dy, const double *preact, double *dx)
{
    const double inv_sqrt2 = 0.70710678118654752440;
    const double inv_sqrt2pi = 0.39894228040143267794;
    for (int64_t i = 0; i < n; ++i) {
        const double x = preact[i];
        const double cdf = 0.5 * erfc(-x * inv_sqrt2);
        const double pdf = inv_sqrt2pi * exp(-0.5 * x * x);
        dx[i] = dy[i] * (cdf + x * pdf);
    }
}

/* The forwards the backward differentiates (for the oracle's own checks). */
void oracle_silu_fwd(int64_t n, const double *x, double *y)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = x[i] / (1.0 + exp(-x[i]));
}

void oracle_gelu_fwd(int64_t n, const double *x, double *y)
{
    const double inv_sqrt2 = 0.70710678118654752440;
    for (int64_t i = 0; i < n; ++i)
        y[i] = x[i] * 0.5 * erfc(-x[i] * inv_sqrt2);
}
