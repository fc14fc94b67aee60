/*
 * kda_oracle.c -- plain fp64 CPU oracle for gated delta-rule linear attention
 * with the lower-bounded per-key-channel decay (Kimi Delta Attention style).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark use it. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes is the plain token-by-token definition, with no chunking and
 * no exp(+/-G) rescaling, so a reader can check it by eye:
 *
 *   for every sequence n and head h:
 *     S = h0[n,h]                      (d_k x d_v, zero when h0 is NULL)
 *     for every token t of sequence n:
 *       g_i   = g_min * sigmoid(a_t,i)   per key channel i
 *               ["Demystifying Trillion-Parameter MoE Models", Breakthrough 1 §2:
 *                g = g_min x sigmoid(.), g_min = -5, g in [g_min, 0);
 *                "From Numerical Stability to Load Balancing", §2.2]
 *       S     <- Diag(exp g) S           (forget: each key row decays)
 *       u     =  beta_t (v_t - S^T k_t)  (delta-rule error, on the decayed S)
 *       S     <- S + k_t u^T             (write the key-value outer product)
 *               ["From Numerical Stability to Load Balancing", §2.1: a
 *                fixed-shape state matrix that forgets through a decay factor
 *                and writes key-value outer products; the delta-rule form of
 *                the write is the one named by the "Kimi Delta Attention" /
 *                "Delta networks" passages of "Architecting Long-Context
 *                LLMs", §2.1-2.2]
 *       o_t   =  scale * S^T q_t          (read the state after the write)
 *     h_final[n,h] = S
 *
 * Layouts (all contiguous, row-major, token-major):
 *   q, k, a : [n_tok, H, d_k]     v : [n_tok, H, d_v]     beta : [n_tok, H]
 *   h0, h_final : [n_seq, H, d_k, d_v]                     out : [n_tok, H, d_v]
 *   cu_seqlens : [n_seq + 1], cu_seqlens[0] = 0, non-decreasing.
 *
 * Independent (sequence, head) items run on a pool of POSIX threads; each item
 * is computed by exactly one thread in the order written above, so the result
 * does not depend on the thread count.
 *
 * Compile-time mutants (KDA_ORACLE_MUTANT = 1..6) plant one plausible mistake
 * each; the test suite builds them to prove that its pins catch such mistakes.
 * The default build (no macro) is the oracle.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef KDA_ORACLE_MUTANT
#define KDA_ORACLE_MUTANT 0
#endif

typedef struct {
    const double *q, *k, *v, *a, *beta, *h0;
    const int64_t *cu_seqlens;
    int64_t n_seq, H, dk, dv;
    double g_min, scale;
    double *out, *h_final;
    /* work distribution */
    const int64_t *order; /* item indices, longest sequence first */
    int64_t n_items;
    int64_t next; /* shared counter, guarded by lock */
    pthread_mutex_t lock;
} job_t;

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static void run_item(job_t *J, int64_t item, double *S, double *gam, double *w) {
    const int64_t n = item / J->H, h = item % J->H;
    const int64_t H = J->H, dk = J->dk, dv = J->dv;
    const int64_t t0 = J->cu_seqlens[n], t1 = J->cu_seqlens[n + 1];

    if (J->h0)
        memcpy(S, J->h0 + (n * H + h) * dk * dv, sizeof(double) * dk * dv);
    else
        memset(S, 0, sizeof(double) * dk * dv);

    for (int64_t t = t0; t < t1; ++t) {
        const double *qt = J->q + (t * H + h) * dk;
        const double *kt = J->k + (t * H + h) * dk;
        const double *at = J->a + (t * H + h) * dk;
        const double *vt = J->v + (t * H + h) * dv;
        const double bt = J->beta[t * H + h];
        double *ot = J->out + (t * H + h) * dv;

        /* bounded per-channel log-decay and its factor */
        for (int64_t i = 0; i < dk; ++i) {
#if KDA_ORACLE_MUTANT == 5 /* mutant: bound dropped (g = -sigmoid) */
            gam[i] = exp(-sigmoid(at[i]));
#else
            gam[i] = exp(J->g_min * sigmoid(at[i]));
#endif
        }

#if KDA_ORACLE_MUTANT == 2 /* mutant: output read before the write */
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += gam[i] * S[i * dv + j] * qt[i];
            ot[j] = J->scale * acc;
        }
#endif

#if KDA_ORACLE_MUTANT != 1
        /* S <- Diag(exp g) S */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= gam[i];
#endif

        /* w = S^T k */
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
#if KDA_ORACLE_MUTANT == 3 /* mutant: transposed state read (needs dk == dv) */
            for (int64_t i = 0; i < dk; ++i) acc += S[j * dv + i] * kt[i];
#else
            for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * kt[i];
#endif
            w[j] = acc;
        }

        /* u = beta (v - S^T k);  S <- S + k u^T */
        for (int64_t j = 0; j < dv; ++j) {
#if KDA_ORACLE_MUTANT == 4 /* mutant: sign of the correction flipped */
            w[j] = bt * (vt[j] + w[j]);
#else
            w[j] = bt * (vt[j] - w[j]);
#endif
        }
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * w[j];

#if KDA_ORACLE_MUTANT == 1 /* mutant: decay applied after the write */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= gam[i];
#endif

#if KDA_ORACLE_MUTANT != 2
        /* o = scale * S^T q */
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * qt[i];
#if KDA_ORACLE_MUTANT == 6 /* mutant: output scale dropped */
            ot[j] = acc;
#else
            ot[j] = J->scale * acc;
#endif
        }
#endif
    }

    if (J->h_final)
        memcpy(J->h_final + (n * H + h) * dk * dv, S, sizeof(double) * dk * dv);
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)(J->dk * J->dv));
    double *gam = (double *)malloc(sizeof(double) * (size_t)J->dk);
    double *w = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!S || !gam || !w) {
        free(S); free(gam); free(w);
        return (void *)1;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t idx = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (idx >= J->n_items) break;
        run_item(J, J->order[idx], S, gam, w);
    }
    free(S); free(gam); free(w);
    return NULL;
}

static const int64_t *g_sort_cu; /* qsort context (single call at a time) */
static int64_t g_sort_H;
static int by_length_desc(const void *x, const void *y) {
    int64_t a = *(const int64_t *)x, b = *(const int64_t *)y;
    int64_t la = g_sort_cu[a / g_sort_H + 1] - g_sort_cu[a / g_sort_H];
    int64_t lb = g_sort_cu[b / g_sort_H + 1] - g_sort_cu[b / g_sort_H];
    if (la != lb) return la < lb ? 1 : -1;
    return a < b ? -1 : (a > b);
}

/* Returns 0 on success, 1 on invalid arguments, 2 on allocation failure. */
int kda_oracle_fwd(const double *q, const double *k, const double *v, const double *a,
                   const double *beta, const double *h0, const int64_t *cu_seqlens,
                   int64_t n_seq, int64_t H, int64_t dk, int64_t dv, double g_min,
                   double scale, double *out, double *h_final, int n_threads) {
    if (n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return 1;
    if (cu_seqlens[0] != 0) return 1;
    for (int64_t n = 0; n < n_seq; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    if (cu_seqlens[n_seq] > 0 && (!q || !k || !v || !a || !beta || !out)) return 1;
    if (n_threads < 1) n_threads = 1;

    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.a = a; J.beta = beta; J.h0 = h0;
    J.cu_seqlens = cu_seqlens;
    J.n_seq = n_seq; J.H = H; J.dk = dk; J.dv = dv;
    J.g_min = g_min; J.scale = scale;
    J.out = out; J.h_final = h_final;
    J.n_items = n_seq * H;
    if (J.n_items == 0) return 0;

    int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)J.n_items);
    if (!order) return 2;
    for (int64_t i = 0; i < J.n_items; ++i) order[i] = i;
    g_sort_cu = cu_seqlens;
    g_sort_H = H;
    qsort(order, (size_t)J.n_items, sizeof(int64_t), by_length_desc);
    J.order = order;
    pthread_mutex_init(&J.lock, NULL);

    if (n_threads > J.n_items) n_threads = (int)J.n_items;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    int rc = 0;
    if (!th) {
        rc = 2;
    } else {
        int started = 0;
        for (int i = 1; i < n_threads; ++i) {
            if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
            ++started;
        }
        if (worker(&J) != NULL) rc = 2;
        for (int i = 1; i <= started; ++i) {
            void *r = NULL;
            pthread_join(th[i], &r);
            if (r != NULL) rc = 2;
        }
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    free(order);
    return rc;
}

int kda_oracle_mutant_id(void) { return KDA_ORACLE_MUTANT; }
