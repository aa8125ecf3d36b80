/*
 * gdn_oracle_bwd.c -- fp64 CPU oracle of the gradients of the gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Called by the tests; the product path never links, loads or calls
 * it, and it shares no code with the CUDA kernels.
 *
 * The forward is the recurrence of gdn_oracle.c (per sequence n and value head h, token by token):
 *
 *   Sb_t = Diag(a_t) S_{t-1}            decayed state   (a_t = exp(g_t), or exp(gk_t) per key channel)
 *   r_t  = Sb_t^T k_t                   read-out
 *   d_t  = beta_t (v_t - r_t)           residual
 *   S_t  = Sb_t + k_t d_t^T             write
 *   o_t  = scale S_t^T q_t
 *
 * This file differentiates it by the chain rule, one token at a time in reverse order
 * ("Flash Linear Attention" page, sec. 7: the backward scans time in reverse and recomputes the
 * states; GDN-in-FLA notes, backward: the gradients dq, dk, dv, dbeta, dg, dh0 of
 * chunk_gated_delta_rule_bwd).  With dS the gradient of the loss with respect to S_t (from the
 * tokens after t and from ht), each step is the adjoint of the forward step read bottom-up:
 *
 *   dS   += scale q_t do_t^T;   dq_t = scale S_t do_t
 *   dd    = dS^T k_t;           dk_t = dS d_t          (from k_t d_t^T)
 *   dv_t  = beta_t dd;          dbeta_t = dd . (v_t - r_t)
 *   dr    = -beta_t dd
 *   dSb   = dS + k_t dr^T;      dk_t += Sb_t dr        (from r_t = Sb_t^T k_t)
 *   dg_t  = sum_j dSb[.,j] Sb_t[.,j]   (per key channel; summed over channels for a scalar gate:
 *                                       d/dg of exp(g) S_{t-1} is exactly Sb_t)
 *   dS    = Diag(a_t) dSb       (the gradient with respect to S_{t-1})
 *
 * starting from dS = dht (or 0); dh0 is the last dS.  The states are recomputed, not stored per
 * token: a forward pass keeps one checkpoint every kBlock tokens, and the reverse pass recomputes
 * the decayed states of one block at a time from its checkpoint.  This is only a memory schedule;
 * every gradient is the token-level chain rule above.
 *
 * dq and dk are written per value head ([T_total, HV, K]); with GVA (HV > H) the caller sums the
 * value heads of each query/key head.
 *
 * Layouts as gdn_oracle.c; do like o [T_total, HV, V]; dht like ht [N, HV, K, V] (nullable);
 * dg like g; dbeta like beta; dh0 like h0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { kBlock = 64 };

typedef struct {
    int n_seqs, H, HV, K, V, gate_kind;
    const int64_t *cu;
    const double *q, *k, *v, *g, *beta, *h0, *dout, *dht;
    double scale;
    double *dq, *dk, *dv, *dbeta, *dg, *dh0;
    int next;
    pthread_mutex_t mu;
} gdn_bwd_job;

typedef struct {
    double *ckpt;  /* state at the start of every block */
    double *sb;    /* decayed states of one block, [kBlock][K][V] */
    double *S, *dS, *dSb, *r, *d, *dd, *dr;
} bwd_scratch;

/* S <- Diag(a_t) S for token t of head h */
static void decay(const gdn_bwd_job *J, int64_t t, int h, double *S)
{
    const int K = J->K, V = J->V;
    if (J->gate_kind == 0) {
        const double a = exp(J->g[(size_t)t * J->HV + h]);
        for (size_t i = 0; i < (size_t)K * V; ++i) S[i] *= a;
    } else {
        const double *gt = J->g + ((size_t)t * J->HV + h) * K;
        for (int dk = 0; dk < K; ++dk) {
            const double a = exp(gt[dk]);
            for (int j = 0; j < V; ++j) S[(size_t)dk * V + j] *= a;
        }
    }
}

/* one forward token: S (holding S_{t-1}) becomes S_t; the decayed state is copied to sb if given */
static void step_fwd(const gdn_bwd_job *J, int64_t t, int h, double *S, double *sb, double *r)
{
    const int K = J->K, V = J->V, hq = h / (J->HV / J->H);
    const double *kt = J->k + ((size_t)t * J->H + hq) * K;
    const double *vt = J->v + ((size_t)t * J->HV + h) * V;
    const double b = J->beta[(size_t)t * J->HV + h];
    decay(J, t, h, S);
    if (sb) memcpy(sb, S, (size_t)K * V * sizeof(double));
    for (int j = 0; j < V; ++j) r[j] = 0.0;
    for (int dk = 0; dk < K; ++dk)
        for (int j = 0; j < V; ++j) r[j] += kt[dk] * S[(size_t)dk * V + j];
    for (int j = 0; j < V; ++j) r[j] = b * (vt[j] - r[j]);
    for (int dk = 0; dk < K; ++dk)
        for (int j = 0; j < V; ++j) S[(size_t)dk * V + j] += kt[dk] * r[j];
}

static void run_pair(const gdn_bwd_job *J, int n, int h, bwd_scratch *W)
{
    const int H = J->H, HV = J->HV, K = J->K, V = J->V, hq = h / (HV / H);
    const size_t KV = (size_t)K * V;
    const int64_t t0 = J->cu[n], T = J->cu[n + 1] - t0;
    const int64_t nb = (T + kBlock - 1) / kBlock;

    /* forward: a checkpoint at the start of every block */
    if (J->h0) memcpy(W->S, J->h0 + ((size_t)n * HV + h) * KV, KV * sizeof(double));
    else memset(W->S, 0, KV * sizeof(double));
    for (int64_t b = 0; b < nb; ++b) {
        memcpy(W->ckpt + (size_t)b * KV, W->S, KV * sizeof(double));
        const int64_t e = (b + 1) * kBlock < T ? (b + 1) * kBlock : T;
        for (int64_t i = b * kBlock; i < e; ++i) step_fwd(J, t0 + i, h, W->S, NULL, W->r);
    }

    /* reverse */
    if (J->dht) memcpy(W->dS, J->dht + ((size_t)n * HV + h) * KV, KV * sizeof(double));
    else memset(W->dS, 0, KV * sizeof(double));
    for (int64_t b = nb - 1; b >= 0; --b) {
        const int64_t s = b * kBlock, e = (b + 1) * kBlock < T ? (b + 1) * kBlock : T;
        /* the block's decayed states from its checkpoint */
        memcpy(W->S, W->ckpt + (size_t)b * KV, KV * sizeof(double));
        for (int64_t i = s; i < e; ++i) step_fwd(J, t0 + i, h, W->S, W->sb + (size_t)(i - s) * KV, W->r);
        for (int64_t i = e - 1; i >= s; --i) {
            const int64_t t = t0 + i;
            const double *sb = W->sb + (size_t)(i - s) * KV;
            const double *qt = J->q + ((size_t)t * H + hq) * K;
            const double *kt = J->k + ((size_t)t * H + hq) * K;
            const double *vt = J->v + ((size_t)t * HV + h) * V;
            const double *dot = J->dout + ((size_t)t * HV + h) * V;
            const double b_ = J->beta[(size_t)t * HV + h];
            double *dqt = J->dq + ((size_t)t * HV + h) * K;
            double *dkt = J->dk + ((size_t)t * HV + h) * K;
            double *dvt = J->dv + ((size_t)t * HV + h) * V;
            /* r = Sb^T k, d = beta (v - r), S_t = Sb + k d^T */
            for (int j = 0; j < V; ++j) W->r[j] = 0.0;
            for (int dk = 0; dk < K; ++dk)
                for (int j = 0; j < V; ++j) W->r[j] += kt[dk] * sb[(size_t)dk * V + j];
            for (int j = 0; j < V; ++j) W->d[j] = b_ * (vt[j] - W->r[j]);
            for (int dk = 0; dk < K; ++dk)
                for (int j = 0; j < V; ++j) W->S[(size_t)dk * V + j] = sb[(size_t)dk * V + j] + kt[dk] * W->d[j];
            /* o_t = scale S_t^T q_t */
            for (int dk = 0; dk < K; ++dk) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) {
                    W->dS[(size_t)dk * V + j] += J->scale * qt[dk] * dot[j];
                    acc += W->S[(size_t)dk * V + j] * dot[j];
                }
                dqt[dk] = J->scale * acc;
            }
            /* S_t = Sb + k d^T */
            for (int j = 0; j < V; ++j) W->dd[j] = 0.0;
            for (int dk = 0; dk < K; ++dk) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) {
                    W->dd[j] += W->dS[(size_t)dk * V + j] * kt[dk];
                    acc += W->dS[(size_t)dk * V + j] * W->d[j];
                }
                dkt[dk] = acc;
            }
            /* d = beta (v - r) */
            double db = 0.0;
            for (int j = 0; j < V; ++j) {
                dvt[j] = b_ * W->dd[j];
                db += W->dd[j] * (vt[j] - W->r[j]);
                W->dr[j] = -b_ * W->dd[j];
            }
            J->dbeta[(size_t)t * HV + h] = db;
            /* r = Sb^T k:  dSb = dS + k dr^T, dk += Sb dr */
            for (int dk = 0; dk < K; ++dk) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) {
                    W->dSb[(size_t)dk * V + j] = W->dS[(size_t)dk * V + j] + kt[dk] * W->dr[j];
                    acc += sb[(size_t)dk * V + j] * W->dr[j];
                }
                dkt[dk] += acc;
            }
            /* Sb = Diag(exp g) S_{t-1}: dg = <dSb, Sb> (per key channel), dS_{t-1} = Diag(exp g) dSb */
            if (J->gate_kind == 0) {
                double acc = 0.0;
                for (size_t x = 0; x < KV; ++x) acc += W->dSb[x] * sb[x];
                J->dg[(size_t)t * HV + h] = acc;
                const double a = exp(J->g[(size_t)t * HV + h]);
                for (size_t x = 0; x < KV; ++x) W->dS[x] = a * W->dSb[x];
            } else {
                const double *gt = J->g + ((size_t)t * HV + h) * K;
                double *dgt = J->dg + ((size_t)t * HV + h) * K;
                for (int dk = 0; dk < K; ++dk) {
                    const double a = exp(gt[dk]);
                    double acc = 0.0;
                    for (int j = 0; j < V; ++j) {
                        acc += W->dSb[(size_t)dk * V + j] * sb[(size_t)dk * V + j];
                        W->dS[(size_t)dk * V + j] = a * W->dSb[(size_t)dk * V + j];
                    }
                    dgt[dk] = acc;
                }
            }
        }
    }
    if (J->dh0) memcpy(J->dh0 + ((size_t)n * HV + h) * KV, W->dS, KV * sizeof(double));
}

static void *worker(void *arg)
{
    gdn_bwd_job *J = (gdn_bwd_job *)arg;
    const size_t KV = (size_t)J->K * J->V;
    int64_t maxlen = 0;
    for (int n = 0; n < J->n_seqs; ++n)
        if (J->cu[n + 1] - J->cu[n] > maxlen) maxlen = J->cu[n + 1] - J->cu[n];
    const size_t nb = (size_t)((maxlen + kBlock - 1) / kBlock) + 1;
    bwd_scratch W;
    W.ckpt = (double *)malloc(nb * KV * sizeof(double));
    W.sb = (double *)malloc((size_t)kBlock * KV * sizeof(double));
    W.S = (double *)malloc(KV * sizeof(double));
    W.dS = (double *)malloc(KV * sizeof(double));
    W.dSb = (double *)malloc(KV * sizeof(double));
    W.r = (double *)malloc((size_t)J->V * sizeof(double));
    W.d = (double *)malloc((size_t)J->V * sizeof(double));
    W.dd = (double *)malloc((size_t)J->V * sizeof(double));
    W.dr = (double *)malloc((size_t)J->V * sizeof(double));
    void *rc = NULL;
    if (!W.ckpt || !W.sb || !W.S || !W.dS || !W.dSb || !W.r || !W.d || !W.dd || !W.dr) {
        rc = (void *)1;
    } else {
        for (;;) {
            pthread_mutex_lock(&J->mu);
            const int idx = J->next++;
            pthread_mutex_unlock(&J->mu);
            if (idx >= J->n_seqs * J->HV) break;
            run_pair(J, idx / J->HV, idx % J->HV, &W);
        }
    }
    free(W.ckpt); free(W.sb); free(W.S); free(W.dS); free(W.dSb);
    free(W.r); free(W.d); free(W.dd); free(W.dr);
    return rc;
}

/*
 * Returns 0 on success, -1 on invalid arguments, -2 on allocation/thread failure.
 * dq, dk: [T_total, HV, K] (per value head).  nthreads <= 0 means one thread.
 */
int gdn_oracle_backward(int n_seqs, const int64_t *cu, int H, int HV, int K, int V, int gate_kind,
                        const double *q, const double *k, const double *v, const double *g,
                        const double *beta, double scale, const double *h0, const double *dout,
                        const double *dht, double *dq, double *dk, double *dv, double *dbeta,
                        double *dg, double *dh0, int nthreads)
{
    if (n_seqs < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || HV % H != 0) return -1;
    if (gate_kind != 0 && gate_kind != 1) return -1;
    if (!cu || !q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dbeta || !dg) return -1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu[n + 1] < cu[n]) return -1;

    gdn_bwd_job J;
    J.n_seqs = n_seqs; J.H = H; J.HV = HV; J.K = K; J.V = V; J.gate_kind = gate_kind;
    J.cu = cu; J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0;
    J.dout = dout; J.dht = dht; J.scale = scale;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dbeta = dbeta; J.dg = dg; J.dh0 = dh0; J.next = 0;
    pthread_mutex_init(&J.mu, NULL);

    int pairs = n_seqs * HV;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pairs) nthreads = pairs > 0 ? pairs : 1;
    int rc = 0;
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
    pthread_mutex_destroy(&J.mu);
    return rc;
}
