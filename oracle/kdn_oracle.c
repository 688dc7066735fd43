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
 *  (3) Backward pass of (1) -- the pages' kernels exist for training on GPUs
 *      ("Learning to Remember, Learn, and Forget in Attention-Based Models",
 *      Contributi Chiave).  oracle_diag_scan_bwd is plain reverse-mode
 *      differentiation of the loop of (1), statement by statement, for the
 *      scalar  L = sum dout . o + sum dmu_T . mu_T + sum dI_T . I_T:
 *      every state of every token is kept, and the chain rule is applied to
 *      the two update statements and the readout in reverse order.  The
 *      outputs are dL/dq, dL/dk, dL/dv, dL/dbeta, dL/dd, dL/dA (per (b,h),
 *      summed over b by the caller), dL/dI_0 and dL/dmu_0.  I_prior is a
 *      fixed hyperparameter here and gets no gradient.
 *
 *  (4) The non-metaplastic limit of (1) ("Learning to Remember, Learn, and
 *      Forget in Attention-Based Models", Metodologia 4, Unificazione
 *      Teorica: Mamba2 is the case where the importance stays at I_prior).
 *      oracle_lin_scan holds I_t = I_{t-1} = I_prior in the mean update of
 *      (1), which leaves
 *          mu_t = alpha_t mu_{t-1} + (1 / I_prior) . [(beta_t . v_t) (x) k_t]
 *      with the same readout o_t[i] = sum_j mu_t[i][j] q_t[j].
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

/* The non-metaplastic limit ((4) in the header).  mu0 and mu_T may be NULL
 * (mu_0 = 0; no final state). */
int oracle_lin_scan(const double* q, const double* k, const double* v,
                    const double* beta, const double* d, const double* A,
                    double I_prior, const double* mu0, double* out, double* mu_T,
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
        if (!mu) {
            failed = 1;
            continue;
        }
        for (long e = 0; e < dv * dk; ++e) mu[e] = mu0 ? mu0[bh * dv * dk + e] : 0.0;
        for (long t = 0; t < T; ++t) {
            const double* qt = q + (bh * T + t) * dk;
            const double* kt = k + (bh * T + t) * dk;
            const double* vt = v + (bh * T + t) * dv;
            const double* bt = beta + (bh * T + t) * dv;
            double alpha = exp(-A[h] * d[bh * T + t]);
            for (long i = 0; i < dv; ++i)
                for (long j = 0; j < dk; ++j) {
                    long e = i * dk + j;
                    /* mu_t = alpha mu_{t-1} + (1/I_prior) (beta_i v_i) k_j */
                    mu[e] = alpha * mu[e] + (1.0 / I_prior) * ((bt[i] * vt[i]) * kt[j]);
                }
            double* ot = out + (bh * T + t) * dv;
            for (long i = 0; i < dv; ++i) {
                double s = 0.0;
                for (long j = 0; j < dk; ++j) s += mu[i * dk + j] * qt[j];
                ot[i] = s;
            }
        }
        if (mu_T)
            for (long e = 0; e < dv * dk; ++e) mu_T[bh * dv * dk + e] = mu[e];
        free(mu);
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

/* Reverse-mode derivative of oracle_diag_scan (see (3) in the header).
 * dout: [B,H,T,dv]; dmu_T, dI_T: [B,H,dv,dk] or NULL (zero).
 * Outputs (all written): dq, dk: [B,H,T,dk]; dv, dbeta: [B,H,T,dv];
 * dd: [B,H,T]; dA_bh: [B,H] (the head's dA contribution of batch b);
 * dI0, dmu0: [B,H,dv,dk] (gradients of the initial state actually used).
 * Memory: (T+1) * dv * dk * 2 doubles per head in flight. */
int oracle_diag_scan_bwd(const double* q, const double* k, const double* v,
                         const double* beta, const double* d, const double* A,
                         double I_prior, const double* I0, const double* mu0,
                         const double* dout, const double* dmu_T, const double* dI_T,
                         double* dq, double* dk_out, double* dv_out, double* dbeta,
                         double* dd, double* dA_bh, double* dI0, double* dmu0,
                         long B, long H, long T, long dk, long dv) {
    if (B < 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return -1;
    long BH = B * H;
    long S = dv * dk;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long bh = 0; bh < BH; ++bh) {
        long h = bh % H;
        /* Is[t], Ms[t]: I and mu after token t (t = 0: the initial state) */
        double* Is = (double*)malloc(sizeof(double) * (T + 1) * S);
        double* Ms = (double*)malloc(sizeof(double) * (T + 1) * S);
        double* gI = (double*)malloc(sizeof(double) * S);
        double* gM = (double*)malloc(sizeof(double) * S);
        if (!Is || !Ms || !gI || !gM) {
            failed = 1;
            free(Is);
            free(Ms);
            free(gI);
            free(gM);
            continue;
        }
        /* ---- forward: the loop of oracle_diag_scan, keeping every state ---- */
        for (long e = 0; e < S; ++e) {
            Is[e] = I0 ? I0[bh * S + e] : I_prior;
            Ms[e] = mu0 ? mu0[bh * S + e] : 0.0;
        }
        for (long t = 0; t < T; ++t) {
            const double* kt = k + (bh * T + t) * dk;
            const double* vt = v + (bh * T + t) * dv;
            const double* bt = beta + (bh * T + t) * dv;
            double alpha = exp(-A[h] * d[bh * T + t]);
            const double* Ip = Is + t * S;
            const double* Mp = Ms + t * S;
            double* In = Is + (t + 1) * S;
            double* Mn = Ms + (t + 1) * S;
            for (long i = 0; i < dv; ++i)
                for (long j = 0; j < dk; ++j) {
                    long e = i * dk + j;
                    In[e] = alpha * Ip[e] + (1.0 - alpha) * I_prior + bt[i] * (kt[j] * kt[j]);
                    Mn[e] = alpha * (Ip[e] / In[e]) * Mp[e] + (1.0 / In[e]) * ((bt[i] * vt[i]) * kt[j]);
                }
        }
        /* ---- reverse: adjoints gI, gM of I_t, mu_t, from t = T down to 1 ---- */
        for (long e = 0; e < S; ++e) {
            gI[e] = dI_T ? dI_T[bh * S + e] : 0.0;
            gM[e] = dmu_T ? dmu_T[bh * S + e] : 0.0;
        }
        double gA = 0.0;
        for (long t = T - 1; t >= 0; --t) {
            const double* qt = q + (bh * T + t) * dk;
            const double* kt = k + (bh * T + t) * dk;
            const double* vt = v + (bh * T + t) * dv;
            const double* bt = beta + (bh * T + t) * dv;
            const double* ot_bar = dout + (bh * T + t) * dv;
            double* dqt = dq + (bh * T + t) * dk;
            double* dkt = dk_out + (bh * T + t) * dk;
            double* dvt = dv_out + (bh * T + t) * dv;
            double* dbt = dbeta + (bh * T + t) * dv;
            double alpha = exp(-A[h] * d[bh * T + t]);
            const double* Ip = Is + t * S;
            const double* Mp = Ms + t * S;
            const double* In = Is + (t + 1) * S;
            const double* Mn = Ms + (t + 1) * S;
            for (long j = 0; j < dk; ++j) dqt[j] = dkt[j] = 0.0;
            for (long i = 0; i < dv; ++i) dvt[i] = dbt[i] = 0.0;
            double g_alpha = 0.0;
            for (long i = 0; i < dv; ++i)
                for (long j = 0; j < dk; ++j) {
                    long e = i * dk + j;
                    /* readout o_t[i] = sum_j mu_t[i][j] q_t[j] */
                    double gmu = gM[e] + ot_bar[i] * qt[j];
                    dqt[j] += ot_bar[i] * Mn[e];
                    /* mu_t = alpha (I_{t-1}/I_t) mu_{t-1} + (1/I_t) (beta_i v_i) k_j */
                    double g_In = gI[e] - gmu * Mn[e] / In[e];
                    g_alpha += gmu * (Ip[e] / In[e]) * Mp[e];
                    double g_Ip = gmu * alpha * Mp[e] / In[e];
                    double g_Mp = gmu * alpha * Ip[e] / In[e];
                    dbt[i] += gmu * vt[i] * kt[j] / In[e];
                    dvt[i] += gmu * bt[i] * kt[j] / In[e];
                    dkt[j] += gmu * bt[i] * vt[i] / In[e];
                    /* I_t = alpha I_{t-1} + (1 - alpha) I_prior + beta_i k_j^2 */
                    g_alpha += g_In * (Ip[e] - I_prior);
                    g_Ip += g_In * alpha;
                    dbt[i] += g_In * kt[j] * kt[j];
                    dkt[j] += g_In * 2.0 * bt[i] * kt[j];
                    gI[e] = g_Ip;
                    gM[e] = g_Mp;
                }
            /* alpha_t = exp(-A d_t) */
            dd[bh * T + t] = g_alpha * (-A[h] * alpha);
            gA += g_alpha * (-d[bh * T + t] * alpha);
        }
        dA_bh[bh] = gA;
        for (long e = 0; e < S; ++e) {
            dI0[bh * S + e] = gI[e];
            dmu0[bh * S + e] = gM[e];
        }
        free(Is);
        free(Ms);
        free(gI);
        free(gM);
    }
    return failed ? -2 : 0;
}
