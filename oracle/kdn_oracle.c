/*
 * kdn_oracle.c -- plain fp64 CPU oracle for the two scans.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may build, load or
 * call it.  It shares no code, header, table or helper with the CUDA
 * library, and the library never calls it.
 *
 * Both functions are literal token-by-token loops over the equations as the
 * pages print them; no blocking, reordering or algebraic rewriting.
 *
 *  (1) Diagonal metaplastic update -- "Learning to Remember, Learn, and
 *      Forget in Attention-Based Models", Metodologia 1 (forget gate
 *      alpha_t = exp(-A d_t)) and Metodologia 2 (the closed-form update of the
 *      importance I_t and the mean mu_t):
 *          I_t  = alpha_t I_{t-1} + (1 - alpha_t) I_prior + beta_t (x) k_t^2
 *          mu_t = alpha_t (I_{t-1} / I_t) . mu_{t-1}
 *                 + (1 / I_t) . [(beta_t . v_t) (x) k_t]
 *      Readout: the output is the posterior mean read through the query
 *      ("Kalman Linear Attention (KLA)", Metodologia 1, "Readout"),
 *          o_t[i] = sum_j mu_t[i][j] q_t[j]        (post-update mu_t).
 *      Readings where the pages are silent: d_t is one scalar per (b,h,t);
 *      A is one scalar per head; beta_t lives on the value axis (d_v) and
 *      (x) is the outer product of a d_v vector with a d_k vector, so
 *      beta_t (x) k_t^2 [i][j] = beta_t[i] k_t[j]^2 and
 *      (beta_t . v_t) (x) k_t [i][j] = beta_t[i] v_t[i] k_t[j];
 *      mu and I are d_v x d_k (row i <-> value, column j <-> key);
 *      I_prior is a scalar; with no initial state given, I_0 = I_prior
 *      and mu_0 = 0.
 *
 *  (2) Moebius precision recursion -- "Kalman Linear Attention (KLA)",
 *      Metodologia 2 ("Parallelizzazione tramite Trasformazioni di
 *      Moebius"), the precision update
 *          lambda_t = (a_t lambda_{t-1} + b_t) / (c_t lambda_{t-1} + d_t)
 *      (the page writes the four coefficients as alpha, beta, gamma, delta;
 *      they are unrelated to the forget gate and importance above).  Step t
 *      uses the coefficients of index t and the output is lambda_1..lambda_T.
 *
 * Parity pins (tests/test_oracle_pins.py) tie every term of these loops to
 * closed forms, special cases and brute force; see that file.
 *
 * Layouts (all row-major, contiguous, fp64):
 *   q, k: [B,H,T,dk]   v, beta: [B,H,T,dv]   d: [B,H,T]   A: [H]
 *   I0, mu0 (optional, may be NULL): [B,H,dv,dk]
 *   out: [B,H,T,dv]    mu_T, I_T (optional, may be NULL): [B,H,dv,dk]
 *   Moebius a, b, c, d, out: [N,T]   lambda0: [N]
 *
 * The only parallelism is an OpenMP loop over independent heads (b,h); each
 * head runs the same sequential loop.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_diag_scan(const double* q, const double* k, const double* v,
                     const double* beta, const double* d, const double* A,
                     double I_prior, const double* I0, const double* mu0,
                     double* out, double* mu_T, double* I_T,
                     long B, long H, long T, long dk, long dv) {
    if (B < 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return -1;
    long BH = B * H;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long bh = 0; bh < BH; ++bh) {
        long h = bh % H;
        double* mu = (double*)malloc(sizeof(double) * dv * dk);
        double* I = (double*)malloc(sizeof(double) * dv * dk);
        if (!mu || !I) {
            failed = 1;
            free(mu);
            free(I);
            continue;
        }
        /* initial state: given, or I_0 = I_prior and mu_0 = 0 */
        for (long e = 0; e < dv * dk; ++e) {
            I[e] = I0 ? I0[bh * dv * dk + e] : I_prior;
            mu[e] = mu0 ? mu0[bh * dv * dk + e] : 0.0;
        }
        for (long t = 0; t < T; ++t) {
            const double* qt = q + (bh * T + t) * dk;
            const double* kt = k + (bh * T + t) * dk;
            const double* vt = v + (bh * T + t) * dv;
            const double* bt = beta + (bh * T + t) * dv;
            /* forget gate alpha_t = exp(-A d_t) */
            double alpha = exp(-A[h] * d[bh * T + t]);
            for (long i = 0; i < dv; ++i) {
                for (long j = 0; j < dk; ++j) {
                    long e = i * dk + j;
                    double I_prev = I[e];
                    /* I_t = alpha I_{t-1} + (1 - alpha) I_prior + beta_i k_j^2 */
                    double I_new = alpha * I_prev + (1.0 - alpha) * I_prior
                                 + bt[i] * (kt[j] * kt[j]);
                    /* mu_t = alpha (I_{t-1}/I_t) mu_{t-1}
                     *        + (1/I_t) (beta_i v_i) k_j */
                    mu[e] = alpha * (I_prev / I_new) * mu[e]
                          + (1.0 / I_new) * ((bt[i] * vt[i]) * kt[j]);
                    I[e] = I_new;
                }
            }
            /* readout with the post-update mean: o_t[i] = sum_j mu[i][j] q_j */
            double* ot = out + (bh * T + t) * dv;
            for (long i = 0; i < dv; ++i) {
                double s = 0.0;
                for (long j = 0; j < dk; ++j) s += mu[i * dk + j] * qt[j];
                ot[i] = s;
            }
        }
        for (long e = 0; e < dv * dk; ++e) {
            if (mu_T) mu_T[bh * dv * dk + e] = mu[e];
            if (I_T) I_T[bh * dv * dk + e] = I[e];
        }
        free(mu);
        free(I);
    }
    return failed ? -2 : 0;
}

int oracle_mobius_scan(const double* a, const double* b, const double* c,
                       const double* d, const double* lambda0, double* out,
                       long N, long T) {
    if (N < 0 || T < 0) return -1;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (long n = 0; n < N; ++n) {
        double lam = lambda0[n];
        for (long t = 0; t < T; ++t) {
            long e = n * T + t;
            /* lambda_t = (a_t lambda_{t-1} + b_t) / (c_t lambda_{t-1} + d_t) */
            lam = (a[e] * lam + b[e]) / (c[e] * lam + d[e]);
            out[e] = lam;
        }
    }
    return 0;
}
