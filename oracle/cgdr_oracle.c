/*
 * cgdr_oracle.c -- fp64 CPU oracle for the channelwise gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (the plain definition, token by token, no blocking and no
 * fusion).  Sources:
 *   - "Two-pass optimization for channelwise gated delta rule kernel"
 *     (executorch PR #21020), Summary: per token the state is decayed, the
 *     value is predicted from the decayed state, a rank-one correction is
 *     applied and the output is read from the updated state.  The PR fuses
 *     these into two traversals; this oracle keeps all four, one loop each,
 *     because it is meant to be checked by eye, not to be fast.
 *   - "Add fused GatedDeltaNet decode Triton kernel" (executorch PR #18865),
 *     description: Q/K/V split, L2 normalisation of q and k, k-head repeat to
 *     the v-head count and the gating computation of the scalar
 *     GatedDeltaNet gate, g = -exp(A_log) * softplus(a + dt_bias) and
 *     beta = sigmoid(b).
 *
 * For one (batch b, v-head h) and each token t in order:
 *   qn = q / sqrt(sum q^2 + eps) * q_scale      (q_scale default 1/sqrt(dk))
 *   kn = k / sqrt(sum k^2 + eps)
 *   alpha_i = exp(g_i)                           (channelwise log-decay g)
 *   S   <- Diag(alpha) S                         (decay)
 *   vh  =  S^T kn                                (prediction)
 *   S   <- S + beta kn (v - vh)^T                (rank-one correction)
 *   o   =  S^T qn                                (readout after the update)
 * The v-head h reads q/k head floor(h / (Hv/Hk)) (repeat-interleave; the
 * pages only say "head repeat", so this mapping is a convention).
 *
 * Inputs are contiguous fp64 arrays (the caller upcasts bf16/fp32 values
 * exactly):  q,k [B,T,Hk,dk]  v [B,T,Hv,dv]  g [B,T,Hv,dk]  beta [B,T,Hv]
 *            a,b [B,T,Hv]  A_log,dt_bias [Hv]  S0 [B,Hv,dk,dv] (or NULL)
 * Outputs:   o [B,T,Hv,dv]  S [B,Hv,dk,dv]   (fp64)
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int B, T, Hk, Hv, dk, dv;
    int gate_mode;     /* 0: per-channel g and beta given; 1: scalar GatedDeltaNet gate */
    int l2norm;        /* 1: L2-normalise q and k */
    double q_scale;    /* multiplies q after normalisation; <= 0 means 1/sqrt(dk) */
    double eps;        /* added to the sum of squares inside the square root */
    const double *q, *k, *v;
    const double *g, *beta;
    const double *a, *b, *A_log, *dt_bias;
    const double *S0;
    double *o, *S;
    int n_threads;
} cgdr_oracle_args;

/* softplus(x) = log(1 + e^x); above 20 it returns x (the usual threshold). */
static double oracle_softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }
static double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static void run_unit(const cgdr_oracle_args *A, int bi, int h, double *work) {
    const int T = A->T, Hk = A->Hk, Hv = A->Hv, dk = A->dk, dv = A->dv;
    const int rep = Hv / Hk;
    const int hk = h / rep;
    double *qn = work, *kn = work + dk, *alpha = work + 2 * dk, *vh = work + 3 * dk;
    double *S = A->S + ((size_t)bi * Hv + h) * (size_t)dk * dv;
    const double qs = A->q_scale > 0.0 ? A->q_scale : 1.0 / sqrt((double)dk);

    if (A->S0)
        memcpy(S, A->S0 + ((size_t)bi * Hv + h) * (size_t)dk * dv, sizeof(double) * dk * dv);
    else
        memset(S, 0, sizeof(double) * dk * dv);

    for (int t = 0; t < T; ++t) {
        const size_t tok_k = ((size_t)bi * T + t) * Hk + hk;
        const size_t tok_v = ((size_t)bi * T + t) * Hv + h;
        const double *q = A->q + tok_k * dk;
        const double *k = A->k + tok_k * dk;
        const double *v = A->v + tok_v * dv;

        /* L2 normalisation of q and k, then the q scale. */
        double sq = 0.0, sk = 0.0;
        for (int i = 0; i < dk; ++i) { sq += q[i] * q[i]; sk += k[i] * k[i]; }
        const double rq = A->l2norm ? 1.0 / sqrt(sq + A->eps) : 1.0;
        const double rk = A->l2norm ? 1.0 / sqrt(sk + A->eps) : 1.0;
        for (int i = 0; i < dk; ++i) { qn[i] = q[i] * rq * qs; kn[i] = k[i] * rk; }

        /* Gate: per-channel log-decay g and write strength beta. */
        double beta;
        if (A->gate_mode == 0) {
            const double *g = A->g + tok_v * dk;
            for (int i = 0; i < dk; ++i) alpha[i] = exp(g[i]);
            beta = A->beta[tok_v];
        } else {
            const double gs = -exp(A->A_log[h]) * oracle_softplus(A->a[tok_v] + A->dt_bias[h]);
            for (int i = 0; i < dk; ++i) alpha[i] = exp(gs);
            beta = oracle_sigmoid(A->b[tok_v]);
        }

        /* Traversal 1: decay. */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= alpha[i];
        /* Traversal 2: prediction from the decayed state. */
        for (int j = 0; j < dv; ++j) vh[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) vh[j] += S[(size_t)i * dv + j] * kn[i];
        /* Traversal 3: rank-one correction. */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += beta * kn[i] * (v[j] - vh[j]);
        /* Traversal 4: readout from the updated state. */
        double *o = A->o + tok_v * dv;
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) o[j] += S[(size_t)i * dv + j] * qn[i];
    }
}

typedef struct {
    const cgdr_oracle_args *A;
    int first, step;
} worker_arg;

static void *worker(void *p) {
    worker_arg *w = (worker_arg *)p;
    const cgdr_oracle_args *A = w->A;
    double *work = (double *)malloc(sizeof(double) * (3 * (size_t)A->dk + A->dv));
    if (!work) return (void *)1;
    const int units = A->B * A->Hv;
    for (int u = w->first; u < units; u += w->step) run_unit(A, u / A->Hv, u % A->Hv, work);
    free(work);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation/thread failure. */
int cgdr_oracle_recurrence(const cgdr_oracle_args *A) {
    if (!A || A->B < 0 || A->T < 0 || A->Hk <= 0 || A->Hv <= 0 || A->dk <= 0 || A->dv <= 0) return -1;
    if (A->Hv % A->Hk) return -1;
    if (!A->q || !A->k || !A->v || !A->o || !A->S) return -1;
    if (A->gate_mode == 0 && (!A->g || !A->beta)) return -1;
    if (A->gate_mode == 1 && (!A->a || !A->b || !A->A_log || !A->dt_bias)) return -1;
    if (A->gate_mode != 0 && A->gate_mode != 1) return -1;
    const int units = A->B * A->Hv;
    int nt = A->n_threads > 0 ? A->n_threads : 1;
    if (nt > units) nt = units > 0 ? units : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    worker_arg *wa = (worker_arg *)malloc(sizeof(worker_arg) * nt);
    if (!th || !wa) { free(th); free(wa); return -2; }
    int started = 0, rc = 0;
    for (int i = 0; i < nt; ++i) {
        wa[i].A = A; wa[i].first = i; wa[i].step = nt;
        if (pthread_create(&th[i], NULL, worker, &wa[i]) != 0) break;
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret) rc = -2;
    }
    /* Units never handed to a thread (thread creation failed) are run here. */
    if (started < nt) {
        worker_arg rest = {A, started, nt};
        for (int i = started; i < nt; ++i) { rest.first = i; if (worker(&rest)) rc = -2; }
    }
    free(th); free(wa);
    return rc;
}
