/*
 * vla_oracle.c -- plain fp64 CPU reference ("the oracle") for the forward
 * recurrence of Variational Linear Attention (VLA).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file's library.  It shares no
 * code, header, table or constant with the CUDA path.
 *
 * Source: "Variational Linear Attention: Stable Associative Memory for
 * Long-Context Transformers" (V. Pandey, G. Singh; web summary pages in
 * zh/nl/de/es, identical formulas).  Sections cited below are the sections of
 * those summaries:
 *   section 2.1  objective, normalised key k_hat
 *   section 2.2  A_t = M_t^{-1} kept exactly by the Sherman-Morrison rank-1
 *                formula; M_t accumulates outer products of the penalty
 *                directions u
 *   section 2.3  recursive rule, steps 1-3, unit-length k_hat and alpha_hat,
 *                ELU+1 "ratio of recurrences" readout
 *
 * Readings where the pages leave a symbol open (each one is also listed with
 * its reason in the design notes of this repository):
 *   z_t      = A_{t-1} u_t  (the only choice that makes step 1 the
 *              Sherman-Morrison update of M_t = M_{t-1} + u_t u_t^T)
 *   A_0      = lambda0^{-1} I   (M_0 = lambda0 I), unless A0 is given
 *   S_0 = 0, n_0 = 0 unless given
 *   eps      = 1e-6: k_hat = k / max(|k|, eps), alpha_hat = g / max(|g|, eps),
 *              readout denominator phi(q)^T n_t + eps
 *   readout  phi(x) = ELU(x) + 1 elementwise; n_t = n_{t-1} + phi(k_hat_t);
 *            o_t = S_t phi(q_t) / (phi(q_t)^T n_t + eps)   (read after write)
 *
 * Every step is written out literally, token by token, in the order the
 * pages give it: A is updated first, the gate is then formed from the
 * UPDATED A_t as a fresh matrix-vector product, and so on.  No blocking,
 * fusion or reordering.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define VLA_ORACLE_EPS 1e-6

/* flags */
#define ORACLE_FLAG_UNNORMALISED_GATE 1 /* alpha_t = A_t k_hat_t (no unit scaling):
                                           the recursive-least-squares form */

typedef struct {
    const double *q, *k, *v, *u;
    int T, d;
    double lambda0;
    const double *S0, *A0, *n0;
    double *o, *S_T, *A_T, *n_T;
    double *alpha_trace, *snorm_trace, *c_trace;
    int flags;
} head_job;

/* phi(x) = ELU(x) + 1: x + 1 for x > 0, exp(x) for x <= 0 (section 2.3). */
static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* y = X w for a d x d row-major matrix X. */
static void matvec(const double *X, const double *w, double *y, int d) {
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += X[i * d + j] * w[j];
        y[i] = acc;
    }
}

static double dot(const double *a, const double *b, int d) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += a[i] * b[i];
    return acc;
}

static void run_head(const head_job *J) {
    const int d = J->d, T = J->T;
    double *A = (double *)malloc(sizeof(double) * d * d);
    double *S = (double *)malloc(sizeof(double) * d * d);
    double *n = (double *)malloc(sizeof(double) * d);
    double *khat = (double *)malloc(sizeof(double) * d);
    double *z = (double *)malloc(sizeof(double) * d);
    double *g = (double *)malloc(sizeof(double) * d);
    double *alpha = (double *)malloc(sizeof(double) * d);
    double *Sk = (double *)malloc(sizeof(double) * d);
    double *r = (double *)malloc(sizeof(double) * d);
    double *fq = (double *)malloc(sizeof(double) * d);
    double *num = (double *)malloc(sizeof(double) * d);

    /* initial state: A_0 = lambda0^{-1} I (M_0 = lambda0 I), S_0 = 0, n_0 = 0 */
    for (int i = 0; i < d * d; ++i) {
        A[i] = J->A0 ? J->A0[i] : 0.0;
        S[i] = J->S0 ? J->S0[i] : 0.0;
    }
    if (!J->A0)
        for (int i = 0; i < d; ++i) A[i * d + i] = 1.0 / J->lambda0;
    for (int i = 0; i < d; ++i) n[i] = J->n0 ? J->n0[i] : 0.0;

    for (int t = 0; t < T; ++t) {
        const double *qt = J->q + (size_t)t * d, *kt = J->k + (size_t)t * d;
        const double *vt = J->v + (size_t)t * d, *ut = J->u + (size_t)t * d;

        /* key normalised to unit length (sections 2.1 and 2.3) */
        double kn = sqrt(dot(kt, kt, d));
        double ks = 1.0 / (kn > VLA_ORACLE_EPS ? kn : VLA_ORACLE_EPS);
        for (int i = 0; i < d; ++i) khat[i] = kt[i] * ks;

        /* step 1 (section 2.3): A_t = A_{t-1} - z z^T / (1 + u^T z), z = A_{t-1} u */
        matvec(A, ut, z, d);
        double den = 1.0 + dot(ut, z, d);
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) A[i * d + j] -= z[i] * z[j] / den;

        /* step 2 (section 2.3): alpha_hat = A_t k_hat / |A_t k_hat| */
        matvec(A, khat, g, d);
        double gn = sqrt(dot(g, g, d));
        double gs = (J->flags & ORACLE_FLAG_UNNORMALISED_GATE)
                        ? 1.0
                        : 1.0 / (gn > VLA_ORACLE_EPS ? gn : VLA_ORACLE_EPS);
        for (int i = 0; i < d; ++i) alpha[i] = g[i] * gs;

        /* step 3 (section 2.3): S_t = S_{t-1} + (v - S_{t-1} k_hat) alpha_hat^T */
        matvec(S, khat, Sk, d);
        for (int i = 0; i < d; ++i) r[i] = vt[i] - Sk[i];
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) S[i * d + j] += r[i] * alpha[j];

        /* readout (section 2.3): ratio of recurrences with the ELU+1 map */
        for (int i = 0; i < d; ++i) n[i] += phi(khat[i]);
        for (int i = 0; i < d; ++i) fq[i] = phi(qt[i]);
        matvec(S, fq, num, d);
        double rden = dot(fq, n, d) + VLA_ORACLE_EPS;
        for (int i = 0; i < d; ++i) J->o[(size_t)t * d + i] = num[i] / rden;

        if (J->alpha_trace)
            for (int i = 0; i < d; ++i) J->alpha_trace[(size_t)t * d + i] = alpha[i];
        if (J->c_trace) J->c_trace[t] = dot(alpha, khat, d);
        if (J->snorm_trace) {
            double f = 0.0;
            for (int i = 0; i < d * d; ++i) f += S[i] * S[i];
            J->snorm_trace[t] = sqrt(f);
        }
    }

    memcpy(J->S_T, S, sizeof(double) * d * d);
    memcpy(J->A_T, A, sizeof(double) * d * d);
    if (J->n_T) memcpy(J->n_T, n, sizeof(double) * d);

    free(A); free(S); free(n); free(khat); free(z); free(g); free(alpha);
    free(Sk); free(r); free(fq); free(num);
}

typedef struct {
    head_job *jobs;
    int njobs;
    int next;
    pthread_mutex_t mu;
} pool_t;

static void *worker(void *arg) {
    pool_t *P = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&P->mu);
        int i = P->next++;
        pthread_mutex_unlock(&P->mu);
        if (i >= P->njobs) break;
        run_head(&P->jobs[i]);
    }
    return NULL;
}

/*
 * Runs the recurrence for BH independent (batch, head) units.
 * q, k, v, u : [BH, T, d] fp64, row-major (token-major within a unit)
 * S0, A0     : [BH, d, d] or NULL;  n0 : [BH, d] or NULL
 * o          : [BH, T, d];  S_T, A_T : [BH, d, d];  n_T : [BH, d] or NULL
 * alpha_trace: [BH, T, d] or NULL (the gate actually used at each step)
 * c_trace    : [BH, T] or NULL (alpha_t^T k_hat_t)
 * snorm_trace: [BH, T] or NULL (Frobenius norm of S_t after step t)
 * S is stored with S[i][j] mapping key coordinate j to value coordinate i.
 * Returns 0, or -1 on bad arguments.  nthreads <= 0 means one thread.
 */
int vla_oracle_forward(const double *q, const double *k, const double *v, const double *u,
                       int BH, int T, int d, double lambda0, const double *S0,
                       const double *A0, const double *n0, double *o, double *S_T,
                       double *A_T, double *n_T, double *alpha_trace, double *c_trace,
                       double *snorm_trace, int flags, int nthreads) {
    if (BH < 0 || T < 0 || d <= 0 || !(lambda0 > 0.0)) return -1;
    if (BH == 0) return 0;
    if (!S_T || !A_T || (T > 0 && (!q || !k || !v || !u || !o))) return -1;
    head_job *jobs = (head_job *)calloc((size_t)BH, sizeof(head_job));
    for (int b = 0; b < BH; ++b) {
        size_t tok = (size_t)b * T * d, mat = (size_t)b * d * d;
        head_job *J = &jobs[b];
        J->q = q ? q + tok : NULL; J->k = k ? k + tok : NULL;
        J->v = v ? v + tok : NULL; J->u = u ? u + tok : NULL;
        J->T = T; J->d = d; J->lambda0 = lambda0;
        J->S0 = S0 ? S0 + mat : NULL; J->A0 = A0 ? A0 + mat : NULL;
        J->n0 = n0 ? n0 + (size_t)b * d : NULL;
        J->o = o ? o + tok : NULL; J->S_T = S_T + mat; J->A_T = A_T + mat;
        J->n_T = n_T ? n_T + (size_t)b * d : NULL;
        J->alpha_trace = alpha_trace ? alpha_trace + tok : NULL;
        J->c_trace = c_trace ? c_trace + (size_t)b * T : NULL;
        J->snorm_trace = snorm_trace ? snorm_trace + (size_t)b * T : NULL;
        J->flags = flags;
    }
    if (nthreads <= 1 || BH == 1) {
        for (int b = 0; b < BH; ++b) run_head(&jobs[b]);
    } else {
        if (nthreads > BH) nthreads = BH;
        pool_t P;
        P.jobs = jobs; P.njobs = BH; P.next = 0;
        pthread_mutex_init(&P.mu, NULL);
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &P);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        pthread_mutex_destroy(&P.mu);
        free(th);
    }
    free(jobs);
    return 0;
}
