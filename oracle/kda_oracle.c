/*
 * kda_oracle.c -- fp64 CPU oracle for the gated delta rule forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the plain definition of the method, one token at a
 * time, in double precision, in the order the pages give:
 *
 *   "You Could Have Come Up With Kimi Delta Attention", sec. 4 (KDA update
 *   equations) and the five-line recurrence printed after the DPLR table:
 *       S~_t = S_{t-1} Diag(alpha_t)               forget each key channel
 *       vhat = S~_t k_t                            predict
 *       e_t  = beta_t (v_t - vhat)                 correct
 *       S_t  = S~_t + e_t k_t^T                    write
 *       o_t  = S_t (d_k^{-1/2} q_t)                read (after the write)
 *   with alpha_t = exp(g_t), g_t = log alpha_t <= 0 stored per token.
 *   Gated DeltaNet (sec. 3) is the same with one alpha_t for all channels.
 *
 *   Modular MAX "gated_delta" module: the state is stored transposed,
 *   [slot][value_head][d_k][d_v]; each sequence of a ragged batch reads and
 *   writes its pool slot in place; GQA maps value head h to key head
 *   h / (HV / HK); q and k are L2-normalised before use.
 *
 * Readings taken where the pages are silent: the L2 norm is
 * x / sqrt(sum x^2 + 1e-6); the query scale multiplies the normalised query.
 *
 * Gated DeltaProduct ("Linear attention visualized", Gated Delta Product section and its
 * virtual-sequence table) replaces the single transition per token by n_h of them: token t
 * carries n_h keys, values and gates k_{t,j}, v_{t,j}, beta_{t,j}; the forget step runs
 * once, before the first substep, then the predict / correct / write steps run once per
 * substep in order j = 1..n_h, and the query reads the state after the last one.  With
 * n_h = 1 this is exactly the recurrence above.  (The page defines it on Gated DeltaNet's
 * scalar gate; a per-channel gate is applied the same way, once per token.)
 *
 * With delta_rule = 0 the correction is skipped (e_t = beta_t v_t): the additive
 * write of plain causal linear attention ("From Attention to Learned Memory",
 * sec. 1, S_t = S_{t-1} + v_t k_t^T) and, with the forget step kept, of RetNet,
 * Mamba-2 and Gated Linear Attention ("Linear attention visualized", those
 * sections).  It is pinned against the brute-force causal product and the
 * decayed parallel form, and is the reference for the library's additive-write
 * mode.
 *
 * Work is split over (sequence, value head) pairs with POSIX threads; each
 * pair's arithmetic is a straight sequential loop (no blocking, no
 * reassociation).  Compile without -ffast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0 /* tests build planted-mistake variants with -DORACLE_MUTANT=n */
#endif

typedef struct {
    int num_seqs;
    const int64_t *offsets;
    const int64_t *slot_idx;
    int HK, HV, dk, dv;
    int n_h; /* substeps per token: k, v, beta are [T, n_h, ...], q and g per token */
    const float *q, *k, *v, *beta, *g;
    int per_channel;
    double scale;
    int l2norm;
    int delta_rule;
    double *pool;
    double *o;
    const uint8_t *pair_mask;
    int64_t next_pair; /* shared work counter */
    pthread_mutex_t lock;
} oracle_job;

static void l2_normalise(double *x, int n) {
    double ss = 0.0;
    for (int c = 0; c < n; ++c) ss += x[c] * x[c];
    double inv = 1.0 / sqrt(ss + 1e-6);
    for (int c = 0; c < n; ++c) x[c] *= inv;
}

/* One (sequence, value head) pair: the token loop. */
static void run_pair(const oracle_job *J, int b, int h, double *kn, double *qn, double *vhat,
                     double *e) {
    const int dk = J->dk, dv = J->dv, n_h = J->n_h;
    const int ratio = J->HV / J->HK;
    const int kh = h / ratio;
    double *S = J->pool + ((size_t)J->slot_idx[b] * J->HV + h) * (size_t)dk * dv; /* S[c*dv + j] */
    for (int64_t t = J->offsets[b]; t < J->offsets[b + 1]; ++t) {
        const float *qt = J->q + ((size_t)t * J->HK + kh) * dk;
        for (int c = 0; c < dk; ++c) qn[c] = (double)qt[c];
        if (J->l2norm) l2_normalise(qn, dk);
        for (int c = 0; c < dk; ++c) qn[c] *= J->scale;

        for (int sub = 0; sub < n_h; ++sub) {
            const size_t m = (size_t)t * n_h + sub; /* row of the substep in k, v, beta */
            const float *kt = J->k + (m * J->HK + kh) * dk;
            const float *vt = J->v + (m * J->HV + h) * dv;
            const double bt = (double)J->beta[m * J->HV + h];
            for (int c = 0; c < dk; ++c) kn[c] = (double)kt[c];
            if (J->l2norm) l2_normalise(kn, dk);

            /* 1. forget, once per token: key channel c (row c of the stored state) scales by
             *    alpha[c] */
#if ORACLE_MUTANT == 6
            if (1) { /* planted: the forget step repeated at every substep */
#else
            if (sub == 0) {
#endif
                for (int c = 0; c < dk; ++c) {
                    double gc = J->per_channel ? (double)J->g[((size_t)t * J->HV + h) * dk + c]
                                               : (double)J->g[(size_t)t * J->HV + h];
#if ORACLE_MUTANT == 1
                    double a = exp(-gc); /* planted: wrong sign of the log-decay */
#else
                    double a = exp(gc);
#endif
                    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a;
                }
            }
            /* 2. predict: vhat = S~ k (sum over key channels) */
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * kn[c];
                vhat[j] = acc;
            }
            /* 3. correct */
            for (int j = 0; j < dv; ++j) {
#if ORACLE_MUTANT == 2
                e[j] = bt * (vt[j] + vhat[j]); /* planted: wrong sign of the prediction */
#elif ORACLE_MUTANT == 3
                e[j] = (vt[j] - vhat[j]); /* planted: dropped beta */
#else
                e[j] = J->delta_rule ? bt * ((double)vt[j] - vhat[j]) : bt * (double)vt[j];
#endif
            }
            /* 4. write: S += k e^T */
            for (int c = 0; c < dk; ++c)
                for (int j = 0; j < dv; ++j) {
#if ORACLE_MUTANT == 4
                    S[(size_t)c * dv + j] += qn[c] * e[j]; /* planted: query used as write key */
#else
                    S[(size_t)c * dv + j] += kn[c] * e[j];
#endif
                }
#if ORACLE_MUTANT == 7
            if (sub == 0) break; /* planted: later substeps dropped, read after the first */
#endif
        }
        /* 5. read after the last write: o = S (s q) */
        double *ot = J->o + ((size_t)t * J->HV + h) * dv;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
#if ORACLE_MUTANT == 5
            for (int c = 0; c < dk; ++c) acc += S[(size_t)j * dv + c] * qn[c]; /* planted: transposed state */
#else
            for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * qn[c];
#endif
            ot[j] = acc;
        }
    }
}

static void *worker(void *arg) {
    oracle_job *J = (oracle_job *)arg;
    const int64_t npairs = (int64_t)J->num_seqs * J->HV;
    double *buf = (double *)malloc(sizeof(double) * (size_t)(2 * J->dk + 2 * J->dv));
    if (!buf) return NULL;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t p = J->next_pair++;
        pthread_mutex_unlock(&J->lock);
        if (p >= npairs) break;
        if (J->pair_mask && !J->pair_mask[p]) continue;
        int b = (int)(p / J->HV), h = (int)(p % J->HV);
        run_pair(J, b, h, buf, buf + J->dk, buf + 2 * J->dk, buf + 2 * J->dk + J->dv);
    }
    free(buf);
    return NULL;
}

static int run_job(int num_seqs, const int64_t *offsets, const int64_t *slot_idx, int HK, int HV,
                   int dk, int dv, int n_h, const float *q, const float *k, const float *v,
                   const float *beta, const float *g, int per_channel, double scale, int l2norm,
                   int delta_rule, double *pool, double *o, const uint8_t *pair_mask,
                   int nthreads) {
    if (num_seqs < 0 || HK <= 0 || HV <= 0 || HV % HK != 0 || dk <= 0 || dv <= 0 || n_h < 1)
        return -1;
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.num_seqs = num_seqs; J.offsets = offsets; J.slot_idx = slot_idx;
    J.HK = HK; J.HV = HV; J.dk = dk; J.dv = dv; J.n_h = n_h;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.per_channel = per_channel;
    J.scale = scale; J.l2norm = l2norm; J.delta_rule = delta_rule;
    J.pool = pool; J.o = o; J.pair_mask = pair_mask; J.next_pair = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads == 1) {
        worker(&J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        int started = 0;
        for (int i = 0; i < nthreads; ++i)
            if (pthread_create(&th[started], NULL, worker, &J) == 0) ++started;
        if (started == 0) worker(&J);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/*
 * Runs every (sequence, value head) pair (or those with pair_mask[b*HV+h] != 0).
 *   offsets   [num_seqs+1]      token offsets of each sequence (ragged, token-major)
 *   slot_idx  [num_seqs]        pool slot of each sequence
 *   q, k      [T, HK, dk] fp32  (exact copies of the bf16 inputs when those are bf16)
 *   v         [T, HV, dv] fp32
 *   beta      [T, HV]     fp32
 *   g         [T, HV] (scalar) or [T, HV, dk] (per channel) fp32 log-decay
 *   pool      [num_slots, HV, dk, dv] fp64, read and written in place
 *   o         [T, HV, dv] fp64 output
 * Returns 0, or -1 on bad arguments.
 */
int kda_oracle_run(int num_seqs, const int64_t *offsets, const int64_t *slot_idx, int HK, int HV,
                   int dk, int dv, const float *q, const float *k, const float *v,
                   const float *beta, const float *g, int per_channel, double scale, int l2norm,
                   int delta_rule, double *pool, double *o, const uint8_t *pair_mask,
                   int nthreads) {
    return run_job(num_seqs, offsets, slot_idx, HK, HV, dk, dv, 1, q, k, v, beta, g, per_channel,
                   scale, l2norm, delta_rule, pool, o, pair_mask, nthreads);
}

/*
 * Gated DeltaProduct: as kda_oracle_run with n_h substeps per token, over real tokens.
 *   q         [T, HK, dk]           one query per token
 *   k         [T, n_h, HK, dk]      the substeps' keys, in order
 *   v         [T, n_h, HV, dv]
 *   beta      [T, n_h, HV]
 *   g         [T, HV] or [T, HV, dk] one log-decay per token
 *   o         [T, HV, dv]           one output per token
 */
int kda_oracle_gdp_run(int num_seqs, const int64_t *offsets, const int64_t *slot_idx, int HK,
                       int HV, int dk, int dv, int n_h, const float *q, const float *k,
                       const float *v, const float *beta, const float *g, int per_channel,
                       double scale, int l2norm, double *pool, double *o, int nthreads) {
    return run_job(num_seqs, offsets, slot_idx, HK, HV, dk, dv, n_h, q, k, v, beta, g, per_channel,
                   scale, l2norm, 1, pool, o, NULL, nthreads);
}

int kda_oracle_mutant(void) { return ORACLE_MUTANT; }
