/*
 * gmm_oracle.c -- plain float64 CPU reference for one EM step of a Gaussian
 * mixture with spherical or diagonal covariance, and for the top-m soft
 * assignment of points to components.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle against which the CUDA
 * path is checked.  It shares no code, header, table or helper with the CUDA
 * library; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark load it.  It is deliberately slow and direct: every quantity
 * is computed from its definition in double precision, in the order the
 * method states it, with no blocking, fusion or algebraic re-arrangement.
 *
 * Sources (web pages this method is described on):
 *  [FG2] "Flash-GMM: A Memory-Efficient Kernel for Scalable Soft Clustering",
 *        section 2 (GMM background): mixture density, log-likelihood, the
 *        unnormalised E-step score pi_k N_ik, its normalisation into
 *        responsibilities r_ik, the log-sum-exp trick, and the M-step for
 *        N_k, pi_k, mu_k and the variance (isotropic sigma_k^2 I, footnote 1).
 *  [ML1] "ML0094 GMM vs K-Means", paragraph on the EM algorithm and the
 *        "Mathematical Formulation" list: E-step posterior, M-step mean as a
 *        responsibility-weighted average, covariance as the weighted scatter,
 *        weight as the average responsibility; monotone log-likelihood.
 *  [GX5] "GMMXX" README, "Covariance Coverage" table: a diagonal model keeps
 *        a (K, D) variance array, a spherical model a (K,) array.
 *
 * The display formulas of [FG2] section 2 did not survive text extraction.
 * The readings used here (all standard EM for these covariance families):
 *  - log N(x | mu, diag(s2)) = -1/2 sum_d [ log(2 pi s2_d) + (x_d-mu_d)^2/s2_d ]
 *  - spherical: s2_d = sigma_k^2 for every d
 *  - the new variance is taken about the NEW mean, with a second pass over X
 *  - spherical variance is per dimension: sum_i r_ik ||x_i-mu_k'||^2 / (D N_k)
 *  - after the M-step, s2 <- max(s2, var_floor) + reg_covar
 *  - a component with N_k < 1e-30 is "empty": it keeps its previous mean and
 *    variance and its log-weight becomes -inf
 *  - the returned log-likelihood is evaluated at the INPUT parameters
 *    (it falls out of the E-step), summed over all points.
 *
 * Arrays: X is N x D row-major float (bf16 and integer-valued data are
 * exactly representable in float); parameters are double.  Variances are
 * (K) for spherical and (K x D) for diagonal.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_SPHERICAL 0
#define ORACLE_DIAG 1
#define ORACLE_EMPTY_NK 1e-30

static const double LOG_2PI = 1.8378770664093454835606594728112;

/* Variance of component k in dimension d. */
static double var_of(const double *vars, int cov, int D, int64_t k, int d)
{
    return cov == ORACLE_SPHERICAL ? vars[k] : vars[k * D + d];
}

/*
 * Log of the unnormalised E-step score, log(pi_k N(x | mu_k, Sigma_k)),
 * written in the direct difference form [FG2 s.2; ML1].
 */
static double log_score(const float *x, int D, int cov, int64_t k,
                        const double *log_weights, const double *means,
                        const double *vars)
{
    double s = 0.0;
    for (int d = 0; d < D; ++d) {
        double v = var_of(vars, cov, D, k, d);
        double diff = (double)x[d] - means[k * D + d];
        s += log(v) + LOG_2PI + diff * diff / v;
    }
    return log_weights[k] - 0.5 * s;
}

/*
 * Log-scores of one point against all K components, and their log-sum-exp
 * (the log of the mixture density at x) [FG2 s.2, log-sum-exp trick].
 */
static double point_scores(const float *x, int D, int K, int cov,
                           const double *log_weights, const double *means,
                           const double *vars, double *ell)
{
    double mx = -INFINITY;
    for (int k = 0; k < K; ++k) {
        ell[k] = log_score(x, D, cov, k, log_weights, means, vars);
        if (ell[k] > mx) mx = ell[k];
    }
    if (mx == -INFINITY) return -INFINITY;
    double sum = 0.0;
    for (int k = 0; k < K; ++k) sum += exp(ell[k] - mx);
    return mx + log(sum);
}

static int pick_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of threads the oracle would use for a given request. */
int oracle_threads(int nthreads) { return pick_threads(nthreads); }

/*
 * ell[i*K+k] = log(pi_k N(x_i | mu_k, Sigma_k)),  lse[i] = log sum_k exp(ell)
 * For inspection of single E-step quantities by the tests.
 */
int oracle_log_scores(const float *X, int64_t N, int D, int K, int cov,
                      const double *log_weights, const double *means,
                      const double *vars, double *ell, double *lse,
                      int nthreads)
{
    if (N < 0 || D < 1 || K < 1 || (cov != ORACLE_SPHERICAL && cov != ORACLE_DIAG))
        return -1;
    int nt = pick_threads(nthreads);
#pragma omp parallel for num_threads(nt) schedule(static)
    for (int64_t i = 0; i < N; ++i)
        lse[i] = point_scores(X + i * D, D, K, cov, log_weights, means, vars,
                              ell + i * K);
    return 0;
}

/*
 * One EM iteration [FG2 s.2; ML1]:
 *   E:  r_ik = pi_k N_ik / sum_j pi_j N_ij        (computed in log space)
 *       L    = sum_i log sum_k pi_k N_ik          (at the input parameters)
 *   M:  N_k  = sum_i r_ik,  pi_k' = N_k / N
 *       mu_k' = sum_i r_ik x_i / N_k
 *       diag:      s2_kd' = sum_i r_ik (x_id - mu_kd')^2 / N_k
 *       spherical: s2_k'  = sum_i r_ik ||x_i - mu_k'||^2 / (D N_k)
 *       s2' <- max(s2', var_floor) + reg_covar
 * Outputs may not alias inputs.  Returns 0, or -1 on bad arguments.
 */
int oracle_em_step(const float *X, int64_t N, int D, int K, int cov,
                   const double *log_weights, const double *means,
                   const double *vars, double reg_covar, double var_floor,
                   double *new_log_weights, double *new_means,
                   double *new_vars, double *total_loglik, int nthreads)
{
    if (N < 1 || D < 1 || K < 1 || (cov != ORACLE_SPHERICAL && cov != ORACLE_DIAG))
        return -1;
    const int nt = pick_threads(nthreads);
    const int64_t KD = (int64_t)K * D;
    const int64_t nvar = cov == ORACLE_DIAG ? KD : K;

    /* One private accumulator set per thread, combined in thread order. */
    double *Nk_t = calloc((size_t)nt * K, sizeof(double));
    double *S1_t = calloc((size_t)nt * KD, sizeof(double));
    double *SV_t = calloc((size_t)nt * nvar, sizeof(double));
    double *L_t = calloc((size_t)nt, sizeof(double));
    double *ell_t = malloc((size_t)nt * K * sizeof(double));
    if (!Nk_t || !S1_t || !SV_t || !L_t || !ell_t) {
        free(Nk_t); free(S1_t); free(SV_t); free(L_t); free(ell_t);
        return -2;
    }

    /* Pass 1: E-step, log-likelihood, N_k and sum_i r_ik x_i. */
#pragma omp parallel num_threads(nt)
    {
        int t = 0;
#ifdef _OPENMP
        t = omp_get_thread_num();
#endif
        double *ell = ell_t + (int64_t)t * K;
        double *Nk = Nk_t + (int64_t)t * K;
        double *S1 = S1_t + (int64_t)t * KD;
#pragma omp for schedule(static)
        for (int64_t i = 0; i < N; ++i) {
            const float *x = X + i * D;
            double lse = point_scores(x, D, K, cov, log_weights, means, vars, ell);
            L_t[t] += lse;
            for (int k = 0; k < K; ++k) {
                double r = exp(ell[k] - lse);
                Nk[k] += r;
                for (int d = 0; d < D; ++d) S1[(int64_t)k * D + d] += r * (double)x[d];
            }
        }
    }

    double L = 0.0;
    for (int t = 0; t < nt; ++t) L += L_t[t];
    for (int t = 1; t < nt; ++t) {
        for (int k = 0; k < K; ++k) Nk_t[k] += Nk_t[(int64_t)t * K + k];
        for (int64_t j = 0; j < KD; ++j) S1_t[j] += S1_t[(int64_t)t * KD + j];
    }
    const double *Nk = Nk_t;

    /* New means (an empty component keeps its previous mean). */
    for (int k = 0; k < K; ++k)
        for (int d = 0; d < D; ++d) {
            int64_t j = (int64_t)k * D + d;
            new_means[j] = Nk[k] < ORACLE_EMPTY_NK ? means[j] : S1_t[j] / Nk[k];
        }

    /* Pass 2: responsibility-weighted scatter about the new means. */
#pragma omp parallel num_threads(nt)
    {
        int t = 0;
#ifdef _OPENMP
        t = omp_get_thread_num();
#endif
        double *ell = ell_t + (int64_t)t * K;
        double *SV = SV_t + (int64_t)t * nvar;
#pragma omp for schedule(static)
        for (int64_t i = 0; i < N; ++i) {
            const float *x = X + i * D;
            double lse = point_scores(x, D, K, cov, log_weights, means, vars, ell);
            for (int k = 0; k < K; ++k) {
                double r = exp(ell[k] - lse);
                for (int d = 0; d < D; ++d) {
                    double diff = (double)x[d] - new_means[(int64_t)k * D + d];
                    if (cov == ORACLE_DIAG) SV[(int64_t)k * D + d] += r * diff * diff;
                    else SV[k] += r * diff * diff;
                }
            }
        }
    }
    for (int t = 1; t < nt; ++t)
        for (int64_t j = 0; j < nvar; ++j) SV_t[j] += SV_t[(int64_t)t * nvar + j];

    for (int k = 0; k < K; ++k) {
        int empty = Nk[k] < ORACLE_EMPTY_NK;
        new_log_weights[k] = empty ? -INFINITY : log(Nk[k] / (double)N);
        if (cov == ORACLE_DIAG) {
            for (int d = 0; d < D; ++d) {
                int64_t j = (int64_t)k * D + d;
                double v = empty ? vars[j] : SV_t[j] / Nk[k];
                if (!empty) v = (v > var_floor ? v : var_floor) + reg_covar;
                new_vars[j] = v;
            }
        } else {
            double v = empty ? vars[k] : SV_t[k] / ((double)D * Nk[k]);
            if (!empty) v = (v > var_floor ? v : var_floor) + reg_covar;
            new_vars[k] = v;
        }
    }
    *total_loglik = L;

    free(Nk_t); free(S1_t); free(SV_t); free(L_t); free(ell_t);
    return 0;
}

/*
 * Top-m soft assignment: for every point, the m largest responsibilities
 * r_ik (normalised over all K components) and their component indices, in
 * descending order of r; equal values are ordered by the lower index first.
 * This is the multi-assignment read off the final responsibilities
 * [FG2 s.1 and conclusion: boundary vectors stored in several posting
 * lists].  total_loglik (may be NULL) receives sum_i log p(x_i).
 */
int oracle_topm(const float *X, int64_t N, int D, int K, int cov,
                const double *log_weights, const double *means,
                const double *vars, int m, double *resp_out, int32_t *idx_out,
                double *total_loglik, int nthreads)
{
    if (N < 0 || D < 1 || K < 1 || m < 1 || m > K ||
        (cov != ORACLE_SPHERICAL && cov != ORACLE_DIAG))
        return -1;
    const int nt = pick_threads(nthreads);
    double *ell_t = malloc((size_t)nt * K * sizeof(double));
    char *taken_t = malloc((size_t)nt * K);
    double *L_t = calloc((size_t)nt, sizeof(double));
    if (!ell_t || !taken_t || !L_t) {
        free(ell_t); free(taken_t); free(L_t);
        return -2;
    }
#pragma omp parallel num_threads(nt)
    {
        int t = 0;
#ifdef _OPENMP
        t = omp_get_thread_num();
#endif
        double *ell = ell_t + (int64_t)t * K;
        char *taken = taken_t + (int64_t)t * K;
#pragma omp for schedule(static)
        for (int64_t i = 0; i < N; ++i) {
            double lse = point_scores(X + i * D, D, K, cov, log_weights, means,
                                      vars, ell);
            L_t[t] += lse;
            memset(taken, 0, (size_t)K);
            for (int j = 0; j < m; ++j) {
                int best = -1;
                for (int k = 0; k < K; ++k)
                    if (!taken[k] && (best < 0 || ell[k] > ell[best])) best = k;
                taken[best] = 1;
                resp_out[i * m + j] = exp(ell[best] - lse);
                idx_out[i * m + j] = best;
            }
        }
    }
    if (total_loglik) {
        double L = 0.0;
        for (int t = 0; t < nt; ++t) L += L_t[t];
        *total_loglik = L;
    }
    free(ell_t); free(taken_t); free(L_t);
    return 0;
}
