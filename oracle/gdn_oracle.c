/*
 * gdn_oracle.c -- fp64 CPU oracle of the gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the chunked-prefill forward computes.  It is called by the
 * tests, by the smoke check and by the benchmark's CPU-baseline leg; the
 * product path never links, loads or calls it, and it shares no code with the
 * CUDA kernels.
 *
 * What it computes (per sequence n and value head h, token by token, fp64):
 *
 *   S <- h0[n,h]  (dk x dv, row-major [K][V])  or 0
 *   for each token t of the sequence:
 *       S   <- Diag(a_t) S            a_t = exp(g[t,h])          (scalar gate)
 *                                     a_t,d = exp(gk[t,h,d])      (per-key-channel gate)
 *       S   <- S + beta_t k_t (v_t - S^T k_t)^T       (read -> residual -> write)
 *       o_t <- scale * S^T q_t                        (post-update state)
 *   ht[n,h] <- S
 *
 * This is S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 * o_t = scale * S_t^T q_t: the gated delta-rule recurrence of the FlashQLA
 * blog ("Further optimisation via gate decay", the recurrence restated there,
 * written in the transposed [dv,dk] state layout) and of the GDN-in-FLA notes
 * (forward Step 4, state in [dk,dv] layout).  The decay is applied before the
 * read-out because the chunk form's W carries the inclusive cumulative gate
 * (FlashQLA blog, "Key problems", W_i line; GDN-in-FLA notes, Step 3).  The
 * per-channel form is the KDA generalisation Diag(alpha_t) with alpha_t a
 * vector over the key channels ("KDA source walkthrough", the gk branch of
 * chunk_gated_delta_rule_fwd_h).
 *
 * GVA: the query/key head of value head h is h / (HV / H) (same walkthrough,
 * the i_h // (HV // H) indexing).
 *
 * Layouts (all tightly packed, tokens of all sequences concatenated):
 *   q, k  [T_total, H,  K]      v, o  [T_total, HV, V]
 *   g     [T_total, HV] (scalar) or [T_total, HV, K] (channel)
 *   beta  [T_total, HV]         h0, ht [N, HV, K, V]
 *   cu    [N+1] host int64 token offsets (cu[0] = 0, cu[N] = T_total)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int n_seqs, H, HV, K, V, gate_kind;
    const int64_t *cu;
    const double *q, *k, *v, *g, *beta, *h0;
    double scale;
    double *o, *ht;
    int next;
    pthread_mutex_t mu;
} gdn_oracle_job;

/* One (sequence, value-head) pair, serial over its tokens. */
static void run_pair(const gdn_oracle_job *J, int n, int h, double *S, double *r)
{
    const int H = J->H, HV = J->HV, K = J->K, V = J->V;
    const int hq = h / (HV / H);
    const size_t KV = (size_t)K * V;

    if (J->h0)
        memcpy(S, J->h0 + ((size_t)n * HV + h) * KV, KV * sizeof(double));
    else
        memset(S, 0, KV * sizeof(double));

    for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
        const double *qt = J->q + ((size_t)t * H + hq) * K;
        const double *kt = J->k + ((size_t)t * H + hq) * K;
        const double *vt = J->v + ((size_t)t * HV + h) * V;
        const double b = J->beta[(size_t)t * HV + h];
        double *ot = J->o + ((size_t)t * HV + h) * V;

        /* decay: S <- Diag(a_t) S */
        if (J->gate_kind == 0) {
            const double a = exp(J->g[(size_t)t * HV + h]);
            for (size_t i = 0; i < KV; ++i) S[i] *= a;
        } else {
            const double *gt = J->g + ((size_t)t * HV + h) * K;
            for (int d = 0; d < K; ++d) {
                const double a = exp(gt[d]);
                double *row = S + (size_t)d * V;
                for (int j = 0; j < V; ++j) row[j] *= a;
            }
        }
        /* read-out of the decayed state: r = S^T k_t */
        for (int j = 0; j < V; ++j) r[j] = 0.0;
        for (int d = 0; d < K; ++d) {
            const double kd = kt[d];
            const double *row = S + (size_t)d * V;
            for (int j = 0; j < V; ++j) r[j] += kd * row[j];
        }
        /* residual write: S <- S + beta k (v - r)^T */
        for (int j = 0; j < V; ++j) r[j] = b * (vt[j] - r[j]);
        for (int d = 0; d < K; ++d) {
            const double kd = kt[d];
            double *row = S + (size_t)d * V;
            for (int j = 0; j < V; ++j) row[j] += kd * r[j];
        }
        /* output from the post-update state: o = scale S^T q */
        for (int j = 0; j < V; ++j) ot[j] = 0.0;
        for (int d = 0; d < K; ++d) {
            const double qd = qt[d];
            const double *row = S + (size_t)d * V;
            for (int j = 0; j < V; ++j) ot[j] += qd * row[j];
        }
        for (int j = 0; j < V; ++j) ot[j] *= J->scale;
    }
    if (J->ht)
        memcpy(J->ht + ((size_t)n * HV + h) * KV, S, KV * sizeof(double));
}

static void *worker(void *arg)
{
    gdn_oracle_job *J = (gdn_oracle_job *)arg;
    const size_t KV = (size_t)J->K * J->V;
    double *S = (double *)malloc(KV * sizeof(double));
    double *r = (double *)malloc((size_t)J->V * sizeof(double));
    if (!S || !r) { free(S); free(r); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        const int idx = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (idx >= J->n_seqs * J->HV) break;
        run_pair(J, idx / J->HV, idx % J->HV, S, r);
    }
    free(S);
    free(r);
    return NULL;
}

/*
 * Returns 0 on success, -1 on invalid arguments, -2 on allocation/thread
 * failure.  nthreads <= 0 means one thread.
 */
int gdn_oracle_recurrence(int n_seqs, const int64_t *cu, int H, int HV, int K, int V,
                          int gate_kind, const double *q, const double *k, const double *v,
                          const double *g, const double *beta, double scale,
                          const double *h0, double *o, double *ht, int nthreads)
{
    if (n_seqs < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || HV % H != 0) return -1;
    if (gate_kind != 0 && gate_kind != 1) return -1;
    if (!cu || !q || !k || !v || !g || !beta || !o) return -1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu[n + 1] < cu[n]) return -1;

    gdn_oracle_job J;
    J.n_seqs = n_seqs; J.H = H; J.HV = HV; J.K = K; J.V = V; J.gate_kind = gate_kind;
    J.cu = cu; J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0;
    J.scale = scale; J.o = o; J.ht = ht; J.next = 0;
    pthread_mutex_init(&J.mu, NULL);

    int pairs = n_seqs * HV;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pairs) nthreads = pairs > 0 ? pairs : 1;
    int rc = 0;
    if (nthreads == 1) {
        if (worker(&J) != NULL) rc = -2;
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        if (!th) { pthread_mutex_destroy(&J.mu); return -2; }
        int started = 0;
        for (; started < nthreads; ++started)
            if (pthread_create(&th[started], NULL, worker, &J) != 0) break;
        if (started == 0) rc = -2;
        for (int i = 0; i < started; ++i) {
            void *ret = NULL;
            pthread_join(th[i], &ret);
            if (ret != NULL) rc = -2;
        }
        free(th);
    }
    pthread_mutex_destroy(&J.mu);
    return rc;
}
