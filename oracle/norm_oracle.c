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
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

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

/*
 * Timed mode across host threads, for the CPU baseline only: the rows are
 * split into nthreads contiguous blocks, each thread runs the functions
 * above on its block with its own dgamma / dbeta partial, and the partials
 * are added in thread order.  dx is identical to the single-thread call;
 * dgamma / dbeta differ only in the grouping of the row sums.  Returns 0, or
 * -1 if a thread or a partial buffer could not be created.
 */
struct oracle_block {
    int ln;
    int64_t rows, N;
    const double *dy, *x, *gamma, *mean, *rstd;
    double *dx, *dgamma, *dbeta;
};

static void *oracle_block_run(void *arg)
{
    struct oracle_block *b = (struct oracle_block *)arg;
    if (b->ln)
        oracle_ln_bwd(b->rows, b->N, b->dy, b->x, b->gamma, b->mean, b->rstd, b->dx, b->dgamma, b->dbeta);
    else
        oracle_rms_bwd(b->rows, b->N, b->dy, b->x, b->gamma, b->rstd, b->dx, b->dgamma);
    return 0;
}

static int oracle_bwd_threads(int ln, int64_t M, int64_t N, const double *dy, const double *x,
                              const double *gamma, const double *mean, const double *rstd, double *dx,
                              double *dgamma, double *dbeta, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > M)
        nthreads = M > 0 ? (int)M : 1;
    struct oracle_block *blk = calloc((size_t)nthreads, sizeof *blk);
    pthread_t *tid = calloc((size_t)nthreads, sizeof *tid);
    double *part = calloc((size_t)nthreads * (size_t)N * 2, sizeof(double));
    int rc = (blk && tid && part) ? 0 : -1;
    int started = 0;
    for (int t = 0; rc == 0 && t < nthreads; ++t) {
        const int64_t r0 = M * t / nthreads, r1 = M * (t + 1) / nthreads;
        struct oracle_block *b = &blk[t];
        b->ln = ln;
        b->rows = r1 - r0;
        b->N = N;
        b->dy = dy + r0 * N;
        b->x = x + r0 * N;
        b->gamma = gamma;
        b->mean = ln ? mean + r0 : 0;
        b->rstd = rstd + r0;
        b->dx = dx + r0 * N;
        b->dgamma = part + (size_t)t * N * 2;
        b->dbeta = b->dgamma + N;
        if (pthread_create(&tid[t], 0, oracle_block_run, b) != 0)
            rc = -1;
        else
            ++started;
    }
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], 0);
    if (rc == 0) {
        for (int64_t j = 0; j < N; ++j) {
            double g = 0.0, be = 0.0;
            for (int t = 0; t < nthreads; ++t) {
                g += part[(size_t)t * N * 2 + j];
                be += part[(size_t)t * N * 2 + N + j];
            }
            dgamma[j] = g;
            if (ln)
                dbeta[j] = be;
        }
    }
    free(part);
    free(tid);
    free(blk);
    return rc;
}

int oracle_ln_bwd_threads(int64_t M, int64_t N, const double *dy, const double *x, const double *gamma,
                          const double *mean, const double *rstd, double *dx, double *dgamma, double *dbeta,
                          int nthreads)
{
    return oracle_bwd_threads(1, M, N, dy, x, gamma, mean, rstd, dx, dgamma, dbeta, nthreads);
}

int oracle_rms_bwd_threads(int64_t M, int64_t N, const double *dy, const double *x, const double *gamma,
                           const double *rstd, double *dx, double *dgamma, int nthreads)
{
    return oracle_bwd_threads(0, M, N, dy, x, gamma, 0, rstd, dx, dgamma, 0, nthreads);
}
