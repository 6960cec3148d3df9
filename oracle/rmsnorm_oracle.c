/*
 * RMSNorm (and LayerNorm) forward / backward oracle -- plain, slow, obviously
 * correct CPU code.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Every value is carried in IEEE double (fp64). Inputs arrive already rounded
 * to the I/O dtype (f32 / f16 / bf16 values are exact in fp64), so the only
 * rounding here is fp64 rounding, plus the explicit round-to-nearest-even of
 * oracle_round() where a method step produces a dtype value that later steps
 * consume (the saved `added` of the fused-add forward).
 *
 * Sources (FlyDSL pages):
 *   [I769]  issue #769 "Add rmsnorm backward (+ forward saves rstd)",
 *           sections "Current state" (forward statistic rrms) and
 *           "Math (matches quack rmsnorm_bwd_ref)" (c1, dx, dweight).
 *   [PR800] PR #800 "Add fused-add / residual backward", section
 *           "What's included" (added = x + residual, total = d_added +
 *           dresidual_out, dx == dresidual) and its squashed commit
 *           messages (rstd is fp32 of shape (M,), all reductions fp32).
 *
 * Layout: every [M,N] array is row-major contiguous; gamma, beta, dweight,
 * dgamma, dbeta are [N]; rstd and mean are [M]. Nothing is blocked, fused or reordered beyond the definitions:
 * each sum runs j = 0..N-1 (row sums) or m = 0..M-1 (column sums) in order.
 * OpenMP only splits independent rows (dx) or independent columns (dweight);
 * each column is still summed over m in ascending order, so results do not
 * depend on the thread count.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes, numbered like the I/O dtypes the pages test: f32, f16, bf16 */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/*
 * Round v to the nearest value of a binary floating-point format with p
 * significand bits (implicit bit included), minimum normal exponent emin and
 * largest finite value maxf; ties go to the even significand; values that
 * round past maxf become +-inf. Written from the IEEE 754 definition: find
 * the quantum (spacing of representable values) at v's binade, divide,
 * round to an integer with ties-to-even, multiply back. Division and
 * multiplication by a power of two are exact in fp64 for every format used
 * here, so the only rounding is the rint() step, which is the RNE rule itself.
 */
static double round_format(double v, int p, int emin, double maxf)
{
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    int k;
    frexp(v, &k);          /* |v| = f * 2^k, f in [0.5, 1): leading bit 2^(k-1) */
    int e = k - 1;
    if (e < emin) e = emin; /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, e - (p - 1));
    double r = rint(v / quantum) * quantum;   /* default FP env: ties-to-even */
    if (fabs(r) > maxf) return v > 0 ? INFINITY : -INFINITY;
    return r;
}

double oracle_round1(double v, int dtype)
{
    switch (dtype) {
    case ORC_F32:  return round_format(v, 24, -126, ldexp(2.0 - ldexp(1.0, -23), 127));
    case ORC_F16:  return round_format(v, 11, -14, 65504.0);
    case ORC_BF16: return round_format(v, 8, -126, ldexp(2.0 - ldexp(1.0, -7), 127));
    default:       return NAN;
    }
}

void oracle_round(const double *in, double *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round1(in[i], dtype);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Forward [I769, "Current state"]: per row, rrms = 1/sqrt(mean_j x_j^2 + eps);
 * y_j = x_j * rrms * gamma_j. rstd[m] receives rrms in fp64 (the caller rounds
 * it to fp32 when it plays the role of the saved fp32 rstd of [PR800]).
 */
void oracle_rmsnorm_fwd(const double *x, const double *gamma, double eps,
                        int64_t M, int64_t N, double *y, double *rstd, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const double *xr = x + m * N;
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) ss += xr[j] * xr[j];
        double ms = ss / (double)N;
        double r = 1.0 / sqrt(ms + eps);
        rstd[m] = r;
        for (int64_t j = 0; j < N; ++j) y[m * N + j] = xr[j] * r * gamma[j];
    }
}

/*
 * Fused-add forward [PR800, "What's included"]: added = x + residual is
 * saved as residual_out in the I/O dtype; the statistic and the normalised
 * output are taken from that saved (dtype-rounded) `added`, so that forward
 * and backward see the same input row.
 */
void oracle_fused_add_rmsnorm_fwd(const double *x, const double *residual, const double *gamma,
                                  double eps, int64_t M, int64_t N, int dtype,
                                  double *out, double *residual_out, double *rstd, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = 0; j < N; ++j)
            residual_out[m * N + j] = oracle_round1(x[m * N + j] + residual[m * N + j], dtype);
    }
    oracle_rmsnorm_fwd(residual_out, gamma, eps, M, N, out, rstd, nthreads);
}

/*
 * Backward [I769, "Math"]: per row with x_hat = x * rstd and wdy = dy * gamma,
 *   c1 = (1/N) * sum_j x_hat_j * wdy_j
 *   dx_j = (wdy_j - x_hat_j * c1) * rstd        (+ dres_j in the fused case)
 * and over all rows dweight_j = sum_m dy_mj * x_hat_mj.
 * `rstd` is the saved statistic as given (the backward does not recompute it).
 * dres may be NULL (read as zeros, [PR800]).
 */
static void bwd_core(const double *x, const double *gamma, const double *dy, const double *rstd,
                     const double *dres, int64_t M, int64_t N, double *dx, double *dweight,
                     int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const double r = rstd[m];
        double acc = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double x_hat = x[m * N + j] * r;
            double wdy = dy[m * N + j] * gamma[j];
            acc += x_hat * wdy;
        }
        double c1 = acc / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double x_hat = x[m * N + j] * r;
            double wdy = dy[m * N + j] * gamma[j];
            double d = (wdy - x_hat * c1) * r;
            if (dres) d += dres[m * N + j];
            dx[m * N + j] = d;
        }
    }

    /* dweight: each column summed over m = 0..M-1 in order; columns split
     * into independent contiguous ranges, one per thread. */
    for (int64_t j = 0; j < N; ++j) dweight[j] = 0.0;
#pragma omp parallel
    {
        int64_t t = 0, T = 1;
#ifdef _OPENMP
        t = omp_get_thread_num();
        T = omp_get_num_threads();
#endif
        int64_t j0 = N * t / T, j1 = N * (t + 1) / T;
        for (int64_t m = 0; m < M; ++m) {
            const double r = rstd[m];
            for (int64_t j = j0; j < j1; ++j) {
                double x_hat = x[m * N + j] * r;
                dweight[j] += dy[m * N + j] * x_hat;
            }
        }
    }
}

void oracle_rmsnorm_bwd(const double *x, const double *gamma, const double *dy, const double *rstd,
                        int64_t M, int64_t N, double *dx, double *dweight, int nthreads)
{
    bwd_core(x, gamma, dy, rstd, NULL, M, N, dx, dweight, nthreads);
}

/*
 * Fused-add backward [PR800]: the same dx on the saved `added`, plus
 * dresidual_out when given; the result is both dx and dresidual, so only one
 * array is produced.
 */
void oracle_fused_add_rmsnorm_bwd(const double *added, const double *gamma, const double *dy,
                                  const double *rstd, const double *dresidual_out,
                                  int64_t M, int64_t N, double *dx, double *dweight, int nthreads)
{
    bwd_core(added, gamma, dy, rstd, dresidual_out, M, N, dx, dweight, nthreads);
}

/*
 * LayerNorm forward. The pages leave LayerNorm's formulas to its textbook
 * definition: its backward "mirrors" the RMSNorm one "adding mean handling +
 * dbias", and its forward saves mean and rstd ([I769] "Proposed approach"
 * item 6 and the plan's "PR 5 -- LayerNorm backward"; [I769] status notes on
 * PR #801). Per row:
 *   mean = (1/N) sum_j x_j
 *   var  = (1/N) sum_j (x_j - mean)^2          (biased, divide by N)
 *   rstd = 1/sqrt(var + eps)
 *   y_j  = (x_j - mean) * rstd * gamma_j + beta_j    (beta may be NULL: no bias)
 * mean[m] and rstd[m] receive the fp64 statistics.
 */
void oracle_layernorm_fwd(const double *x, const double *gamma, const double *beta, double eps,
                          int64_t M, int64_t N, double *y, double *mean, double *rstd,
                          int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const double *xr = x + m * N;
        double s = 0.0;
        for (int64_t j = 0; j < N; ++j) s += xr[j];
        double mu = s / (double)N;
        double v = 0.0;
        for (int64_t j = 0; j < N; ++j) v += (xr[j] - mu) * (xr[j] - mu);
        double var = v / (double)N;
        double r = 1.0 / sqrt(var + eps);
        mean[m] = mu;
        rstd[m] = r;
        for (int64_t j = 0; j < N; ++j) {
            double yv = (xr[j] - mu) * r * gamma[j];
            if (beta) yv += beta[j];
            y[m * N + j] = yv;
        }
    }
}

/*
 * LayerNorm backward, the gradient of the forward above with the saved mean
 * and rstd taken as given. Per row, x_hat = (x - mean) * rstd, wdy = dy * gamma:
 *   c1 = (1/N) sum_j x_hat_j * wdy_j
 *   c2 = (1/N) sum_j wdy_j
 *   dx_j = (wdy_j - c2 - x_hat_j * c1) * rstd
 * and over all rows dgamma_j = sum_m dy_mj * x_hat_mj, dbeta_j = sum_m dy_mj.
 */
void oracle_layernorm_bwd(const double *x, const double *gamma, const double *dy,
                          const double *mean, const double *rstd, int64_t M, int64_t N,
                          double *dx, double *dgamma, double *dbeta, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const double mu = mean[m], r = rstd[m];
        double a1 = 0.0, a2 = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double x_hat = (x[m * N + j] - mu) * r;
            double wdy = dy[m * N + j] * gamma[j];
            a1 += x_hat * wdy;
            a2 += wdy;
        }
        double c1 = a1 / (double)N;
        double c2 = a2 / (double)N;
        for (int64_t j = 0; j < N; ++j) {
            double x_hat = (x[m * N + j] - mu) * r;
            double wdy = dy[m * N + j] * gamma[j];
            dx[m * N + j] = (wdy - c2 - x_hat * c1) * r;
        }
    }

    for (int64_t j = 0; j < N; ++j) {
        dgamma[j] = 0.0;
        dbeta[j] = 0.0;
    }
#pragma omp parallel
    {
        int64_t t = 0, T = 1;
#ifdef _OPENMP
        t = omp_get_thread_num();
        T = omp_get_num_threads();
#endif
        int64_t j0 = N * t / T, j1 = N * (t + 1) / T;
        for (int64_t m = 0; m < M; ++m) {
            const double mu = mean[m], r = rstd[m];
            for (int64_t j = j0; j < j1; ++j) {
                double x_hat = (x[m * N + j] - mu) * r;
                dgamma[j] += dy[m * N + j] * x_hat;
                dbeta[j] += dy[m * N + j];
            }
        }
    }
}
