/*
 * Gated DeltaNet (GDN) recurrence -- fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark load it.  It shares no code with the CUDA path.
 *
 * What it computes (Qwen3.8-Next reading notes, jianyuh.github.io,
 * section 2.1 "Gated DeltaNet", the four-line gated delta recurrence):
 * per head, with a matrix state S in R^{dk x dv} (rows indexed by the key
 * dimension, "transposed convention"), for t = 1..T in order
 *
 *     S~  = alpha_t * S_{t-1}                 (decay the whole memory)
 *     e_t = v_t - S~^T k_t                    (what is missing under key k_t)
 *     S_t = S~ + beta_t * k_t e_t^T           (write only the residual)
 *     y_t = S_t^T q_t                         (read with the query, after the write)
 *
 * The decay is applied before the residual is formed, as the equation block
 * of section 2.1 states; the conceptual numpy snippet on the ta-paperlens
 * walkthrough ("Inside GDN: erase before you write") forms e from the
 * undecayed state, which disagrees with the equations for alpha < 1 and is
 * not followed.
 *
 * Layouts (dense, row-major, all fp64 here; the caller upcasts the stored
 * bf16/fp32 values exactly):
 *   q, k        [B, T, Hqk, dk]
 *   v, y        [B, T, Hv,  dv]
 *   alpha, beta [B, T, Hv]
 *   S0, S_T     [B, Hv, dk, dv]   (dv contiguous); S0 may be NULL (= zeros)
 * Value head h reads query/key head h / (Hv / Hqk) (contiguous grouping).
 *
 * Each (b, h) pair is an independent sequential loop; pairs are spread over
 * POSIX threads.  No blocking, fusion or reordering beyond the definition.
 *
 * Channel-wise decay (gdn_oracle_recurrence_cw): the decay gate is a vector
 * alpha_t in (0,1]^dk per value head, layout [B, T, Hv, dk], and the decay
 * step scales row i of the state (key dimension i) by alpha_t[i]:
 *     S~ = diag(alpha_t) S_{t-1}
 * -- the per-channel ("diagonal") gate of Kimi Delta Attention, which the
 * pages name as the same family of fast delta-rule kernels (section 2.1, "Why
 * the delta rule matters").  The other three lines are unchanged.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t B, T;
    int Hqk, Hv, dk, dv;
    int alpha_cw;            /* 1: alpha is [B, T, Hv, dk] (per key channel) */
    const double *q, *k, *v, *alpha, *beta, *S0;
    double *y, *S_T;
    int64_t next;            /* next (b, h) pair to take */
    pthread_mutex_t lock;
} oracle_job;

static void run_head(const oracle_job *J, int64_t b, int hv, double *S, double *e)
{
    const int dk = J->dk, dv = J->dv;
    const int group = J->Hv / J->Hqk;
    const int hk = hv / group;
    const size_t state_elems = (size_t)dk * (size_t)dv;

    if (J->S0)
        memcpy(S, J->S0 + ((size_t)b * J->Hv + hv) * state_elems, state_elems * sizeof(double));
    else
        memset(S, 0, state_elems * sizeof(double));

    for (int64_t t = 0; t < J->T; ++t) {
        const size_t tok = (size_t)b * (size_t)J->T + (size_t)t;
        const double *at = J->alpha + (J->alpha_cw ? (tok * J->Hv + hv) * (size_t)dk : tok * J->Hv + hv);
        const double bt = J->beta[tok * J->Hv + hv];
        const double *kt = J->k + (tok * J->Hqk + hk) * dk;
        const double *qt = J->q + (tok * J->Hqk + hk) * dk;
        const double *vt = J->v + (tok * J->Hv + hv) * dv;
        double *yt = J->y + (tok * J->Hv + hv) * dv;

        /* S~ = alpha_t S_{t-1}, or diag(alpha_t) S_{t-1} per key channel */
        for (int i = 0; i < dk; ++i) {
            const double a = J->alpha_cw ? at[i] : at[0];
            double *row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j)
                row[j] *= a;
        }

        /* e_t = v_t - S~^T k_t :  e[j] = v[j] - sum_i S~[i][j] k[i] */
        for (int j = 0; j < dv; ++j)
            e[j] = vt[j];
        for (int i = 0; i < dk; ++i) {
            const double ki = kt[i];
            const double *row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j)
                e[j] -= row[j] * ki;
        }

        /* S_t = S~ + beta_t k_t e_t^T */
        for (int i = 0; i < dk; ++i) {
            const double w = bt * kt[i];
            double *row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j)
                row[j] += w * e[j];
        }

        /* y_t = S_t^T q_t :  y[j] = sum_i S_t[i][j] q[i] */
        for (int j = 0; j < dv; ++j)
            yt[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double qi = qt[i];
            const double *row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j)
                yt[j] += row[j] * qi;
        }
    }

    if (J->S_T)
        memcpy(J->S_T + ((size_t)b * J->Hv + hv) * state_elems, S, state_elems * sizeof(double));
}

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    double *S = (double *)malloc((size_t)J->dk * (size_t)J->dv * sizeof(double));
    double *e = (double *)malloc((size_t)J->dv * sizeof(double));
    if (!S || !e) {
        free(S);
        free(e);
        return (void *)1;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t p = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (p >= J->B * J->Hv)
            break;
        run_head(J, p / J->Hv, (int)(p % J->Hv), S, e);
    }
    free(S);
    free(e);
    return NULL;
}

/*
 * Returns 0 on success, 1 on invalid arguments, 2 on allocation or thread
 * failure.  y must hold B*T*Hv*dv doubles; S_T (may be NULL) B*Hv*dk*dv.
 */
static int run_all(int64_t B, int64_t T, int Hqk, int Hv, int dk, int dv, int alpha_cw,
                   const double *q, const double *k, const double *v,
                   const double *alpha, const double *beta, const double *S0,
                   double *y, double *S_T, int n_threads)
{
    if (B < 0 || T < 0 || Hqk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hqk != 0)
        return 1;
    if ((B * T > 0) && (!q || !k || !v || !alpha || !beta || !y))
        return 1;
    oracle_job J;
    J.B = B; J.T = T; J.Hqk = Hqk; J.Hv = Hv; J.dk = dk; J.dv = dv; J.alpha_cw = alpha_cw;
    J.q = q; J.k = k; J.v = v; J.alpha = alpha; J.beta = beta; J.S0 = S0;
    J.y = y; J.S_T = S_T;
    J.next = 0;
    pthread_mutex_init(&J.lock, NULL);

    int64_t pairs = B * (int64_t)Hv;
    int nt = n_threads < 1 ? 1 : n_threads;
    if (nt > pairs)
        nt = pairs > 0 ? (int)pairs : 1;
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!th)
        return 2;
    int rc = 0, started = 0;
    for (int i = 0; i < nt; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) {
            rc = 2;
            break;
        }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret)
            rc = 2;
    }
    free(th);
    pthread_mutex_destroy(&J.lock);
    return rc;
}

int gdn_oracle_recurrence(int64_t B, int64_t T, int Hqk, int Hv, int dk, int dv,
                          const double *q, const double *k, const double *v,
                          const double *alpha, const double *beta, const double *S0,
                          double *y, double *S_T, int n_threads)
{
    return run_all(B, T, Hqk, Hv, dk, dv, 0, q, k, v, alpha, beta, S0, y, S_T, n_threads);
}

/* As gdn_oracle_recurrence with alpha of layout [B, T, Hv, dk] (channel-wise decay). */
int gdn_oracle_recurrence_cw(int64_t B, int64_t T, int Hqk, int Hv, int dk, int dv,
                             const double *q, const double *k, const double *v,
                             const double *alpha, const double *beta, const double *S0,
                             double *y, double *S_T, int n_threads)
{
    return run_all(B, T, Hqk, Hv, dk, dv, 1, q, k, v, alpha, beta, S0, y, S_T, n_threads);
}
