/*
 * linattn_oracle.c -- plain fp64 CPU oracle for kernelized linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no code, header, table or helper with the CUDA library and
 * never calls it.
 *
 * Everything is computed in double precision, one token at a time, in the
 * order the pages write the recurrence.  No blocking, chunking or reordering
 * is done; the only parallelism is one thread per independent (batch,
 * kv-head) state stream, which does not change any arithmetic.
 *
 * Sources (page title, section):
 *  - "[Feature] LinearAttention layer for Keras", section "Mathematical
 *    definition" (non-causal and causal forms, eps in the denominator,
 *    current token included), "Feature maps" (elu_plus_one, relu), and
 *    "Streaming State" (key_value_state (B,H,Dk,Dv), key_state (B,H,Dk)).
 *  - "Causal Linear Attention" (running sums S_i, Z_i; update, then read out).
 *  - ONNX-light "LinearAttention" operator: packed [B,T,H*D] layout, GQA
 *    head sharing, update rules linear / gated / delta / gated_delta, scale,
 *    decay layouts (B,T,H_kv) and (B,T,H_kv*d_k), beta layouts (B,T,H_kv)
 *    and (B,T,1).
 *  - Same Keras request, section "Masking": a (batch, sequence) validity
 *    mask.  Causal: an invalid step leaves S and Z as they were and its
 *    output is zero.  Non-causal: invalid keys/values add nothing to the
 *    global sums and invalid query positions give zero output.
 *
 * Parity pins: see tests/test_oracle.py (worked examples of the ONNX page,
 * the 0.2188 figure of "Causal Linear Attention", the O(T^2) brute force,
 * closed forms and invariants).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_FMAP_NONE = 0, ORC_FMAP_ELU_PLUS_ONE = 1, ORC_FMAP_RELU_EPS = 2 };
enum { ORC_RULE_LINEAR = 0, ORC_RULE_GATED = 1, ORC_RULE_DELTA = 2, ORC_RULE_GATED_DELTA = 3 };

typedef struct {
    int64_t B, T;
    int32_t Hq, Hkv, Dk, Dv;
    int32_t feature_map;    /* ORC_FMAP_* */
    int32_t use_normalizer; /* 1: y = num / (phi(q).Z + eps); 0: y = num */
    double eps;             /* normalization_epsilon; also the relu offset */
    double scale;           /* output scale, already resolved by the caller */
    int32_t rule;           /* ORC_RULE_* */
    int32_t decay_per_dim;  /* 0: decay (B,T,Hkv); 1: decay (B,T,Hkv*Dk) */
    int32_t beta_per_head;  /* 1: beta (B,T,Hkv); 0: beta (B,T,1) */
    int32_t nthreads;       /* worker threads over (b, kv-head); <=0 -> 1 */
} orc_params;

/* Feature map, "Feature maps" section of the Keras request:
 *   elu_plus_one: elu(x) + 1 with the ELU slope alpha = 1, i.e. x + 1 for
 *                 x > 0 and exp(x) for x <= 0;
 *   relu:         max(x, 0) + normalization_epsilon;
 *   none:         identity (the ONNX rules apply no feature map). */
static double orc_phi(int fmap, double x, double eps)
{
    switch (fmap) {
    case ORC_FMAP_ELU_PLUS_ONE: return x > 0.0 ? x + 1.0 : exp(x);
    case ORC_FMAP_RELU_EPS:     return (x > 0.0 ? x : 0.0) + eps;
    default:                    return x;
    }
}

typedef struct {
    const orc_params* p;
    const double *q, *k, *v, *decay, *beta, *S0, *Z0;
    const unsigned char* mask; /* (B,T), nonzero = valid; NULL = all valid */
    double *y, *S_out, *Z_out;
    int causal;
    int64_t next;          /* shared work counter over (b, kv-head) */
    pthread_mutex_t lock;
} orc_job;

/* One independent state stream: batch b, kv head hk.  Causal: the
 * recurrence of "Mathematical definition / Causal" (Keras request) and the
 * update rules of the ONNX page, token by token: first the state update,
 * then the read-out for every query head that shares this kv head.
 * Non-causal: the global sums S = sum_j phi(K_j)^T V_j, Z = sum_j phi(K_j),
 * then Y_i = phi(Q_i) S / (phi(Q_i) Z + eps).
 * Masking (Keras request, "Masking"): an invalid causal step is skipped, so
 * S_t = S_{t-1}, Z_t = Z_{t-1} and Y_t = 0 (the where(mask_t, candidate,
 * previous) selection, with the candidate never formed); non-causal, an
 * invalid position is left out of the sums and its output is zero. */
static void orc_stream(orc_job* J, int64_t b, int32_t hk, double* S, double* Z,
                       double* fk, double* fq, double* u)
{
    const orc_params* p = J->p;
    const int64_t T = p->T;
    const int32_t Hq = p->Hq, Hkv = p->Hkv, Dk = p->Dk, Dv = p->Dv;
    const int32_t G = Hq / Hkv; /* query heads per kv head */
    const size_t sdim = (size_t)Dk * Dv;

    if (J->S0) memcpy(S, J->S0 + ((size_t)b * Hkv + hk) * sdim, sdim * sizeof(double));
    else memset(S, 0, sdim * sizeof(double));
    if (J->Z0) memcpy(Z, J->Z0 + ((size_t)b * Hkv + hk) * Dk, Dk * sizeof(double));
    else memset(Z, 0, Dk * sizeof(double));

    if (!J->causal) {
        /* global state over all positions */
        for (int64_t t = 0; t < T; ++t) {
            if (J->mask && !J->mask[b * T + t]) continue; /* invalid key/value */
            const double* kt = J->k + ((size_t)(b * T + t) * Hkv + hk) * Dk;
            const double* vt = J->v + ((size_t)(b * T + t) * Hkv + hk) * Dv;
            for (int32_t i = 0; i < Dk; ++i) fk[i] = orc_phi(p->feature_map, kt[i], p->eps);
            for (int32_t i = 0; i < Dk; ++i) {
                for (int32_t j = 0; j < Dv; ++j) S[(size_t)i * Dv + j] += fk[i] * vt[j];
                Z[i] += fk[i];
            }
        }
    }

    for (int64_t t = 0; t < T; ++t) {
        const size_t tok = (size_t)(b * T + t);
        if (J->mask && !J->mask[tok]) {
            /* invalid step: state kept, zero output for every head of the group */
            for (int32_t r = 0; r < G; ++r) {
                double* yt = J->y + (tok * Hq + hk * G + r) * Dv;
                for (int32_t j = 0; j < Dv; ++j) yt[j] = 0.0;
            }
            continue;
        }
        if (J->causal) {
            const double* kt = J->k + (tok * Hkv + hk) * Dk;
            const double* vt = J->v + (tok * Hkv + hk) * Dv;
            for (int32_t i = 0; i < Dk; ++i) fk[i] = orc_phi(p->feature_map, kt[i], p->eps);

            /* decay (log space): S <- exp(g) * S, row i scaled by exp(g_i)
             * in the per-key-dimension layout */
            if (p->rule == ORC_RULE_GATED || p->rule == ORC_RULE_GATED_DELTA) {
                for (int32_t i = 0; i < Dk; ++i) {
                    double g = p->decay_per_dim ? J->decay[(tok * Hkv + hk) * Dk + i]
                                                : J->decay[tok * Hkv + hk];
                    double a = exp(g);
                    for (int32_t j = 0; j < Dv; ++j) S[(size_t)i * Dv + j] *= a;
                }
            }
            if (p->rule == ORC_RULE_DELTA || p->rule == ORC_RULE_GATED_DELTA) {
                /* S <- S + beta k (x) (v - S^T k), S already decayed */
                double bt = p->beta_per_head ? J->beta[tok * Hkv + hk] : J->beta[tok];
                for (int32_t j = 0; j < Dv; ++j) {
                    double acc = 0.0;
                    for (int32_t i = 0; i < Dk; ++i) acc += S[(size_t)i * Dv + j] * fk[i];
                    u[j] = vt[j] - acc;
                }
                for (int32_t i = 0; i < Dk; ++i)
                    for (int32_t j = 0; j < Dv; ++j) S[(size_t)i * Dv + j] += bt * fk[i] * u[j];
            } else {
                /* S <- S + phi(k) (x) v ;  Z <- Z + phi(k) */
                for (int32_t i = 0; i < Dk; ++i)
                    for (int32_t j = 0; j < Dv; ++j) S[(size_t)i * Dv + j] += fk[i] * vt[j];
            }
            for (int32_t i = 0; i < Dk; ++i) Z[i] += fk[i];
        }

        /* read-out for the G query heads that share kv head hk:
         * query head h uses kv head h / G (contiguous groups) */
        for (int32_t r = 0; r < G; ++r) {
            const int32_t h = hk * G + r;
            const double* qt = J->q + (tok * Hq + h) * Dk;
            double* yt = J->y + (tok * Hq + h) * Dv;
            for (int32_t i = 0; i < Dk; ++i) fq[i] = orc_phi(p->feature_map, qt[i], p->eps);
            double den = 1.0;
            if (p->use_normalizer) {
                den = 0.0;
                for (int32_t i = 0; i < Dk; ++i) den += fq[i] * Z[i];
                den += p->eps;
            }
            for (int32_t j = 0; j < Dv; ++j) {
                double num = 0.0;
                for (int32_t i = 0; i < Dk; ++i) num += fq[i] * S[(size_t)i * Dv + j];
                yt[j] = p->scale * (num / den);
            }
        }
    }

    if (J->S_out) memcpy(J->S_out + ((size_t)b * Hkv + hk) * sdim, S, sdim * sizeof(double));
    if (J->Z_out) memcpy(J->Z_out + ((size_t)b * Hkv + hk) * Dk, Z, Dk * sizeof(double));
}

static void* orc_worker(void* arg)
{
    orc_job* J = (orc_job*)arg;
    const orc_params* p = J->p;
    const int64_t n = p->B * p->Hkv;
    double* S = (double*)malloc(sizeof(double) * (size_t)p->Dk * p->Dv);
    double* Z = (double*)malloc(sizeof(double) * (size_t)p->Dk);
    double* fk = (double*)malloc(sizeof(double) * (size_t)p->Dk);
    double* fq = (double*)malloc(sizeof(double) * (size_t)p->Dk);
    double* u = (double*)malloc(sizeof(double) * (size_t)p->Dv);
    if (S && Z && fk && fq && u) {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            int64_t w = J->next++;
            pthread_mutex_unlock(&J->lock);
            if (w >= n) break;
            orc_stream(J, w / p->Hkv, (int32_t)(w % p->Hkv), S, Z, fk, fq, u);
        }
    }
    free(S); free(Z); free(fk); free(fq); free(u);
    return NULL;
}

static int orc_check(const orc_params* p, int causal, const double* decay, const double* beta)
{
    if (!p || p->B < 0 || p->T < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Dk <= 0 || p->Dv <= 0) return 1;
    if (p->Hq % p->Hkv != 0) return 1; /* q_num_heads must be a multiple of kv_num_heads */
    if (p->rule < ORC_RULE_LINEAR || p->rule > ORC_RULE_GATED_DELTA) return 1;
    if (!causal && p->rule != ORC_RULE_LINEAR) return 1; /* the pages define no non-causal decay/delta */
    if (p->use_normalizer && p->rule != ORC_RULE_LINEAR) return 1; /* normalizer only defined for the sum rule */
    if ((p->rule == ORC_RULE_GATED || p->rule == ORC_RULE_GATED_DELTA) && !decay) return 1;
    if ((p->rule == ORC_RULE_DELTA || p->rule == ORC_RULE_GATED_DELTA) && !beta) return 1;
    return 0;
}

static int orc_run(orc_job* J)
{
    const orc_params* p = J->p;
    int nt = p->nthreads > 0 ? p->nthreads : 1;
    const int64_t n = p->B * p->Hkv;
    if (n < nt) nt = (int)(n > 0 ? n : 1);
    J->next = 0;
    pthread_mutex_init(&J->lock, NULL);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    int started = 0;
    for (int i = 1; i < nt; ++i)
        if (pthread_create(&th[started], NULL, orc_worker, J) == 0) ++started;
    orc_worker(J); /* the calling thread works too */
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J->lock);
    return 0;
}

/* Causal pass over T tokens, optionally continuing from (S0, Z0) (NULL means
 * zeros, as get_initial_state / the ONNX default past_state) and returning
 * the final (S, Z) (NULL means not wanted).  Layouts, all row-major:
 *   q (B,T,Hq,Dk)  k (B,T,Hkv,Dk)  v (B,T,Hkv,Dv)  y (B,T,Hq,Dv)
 *   S (B,Hkv,Dk,Dv)  Z (B,Hkv,Dk)
 *   decay (B,T,Hkv) or (B,T,Hkv,Dk); beta (B,T,Hkv) or (B,T,1).
 *   mask (B,T) validity, nonzero = valid; NULL (orc_causal) = all valid.
 * Returns 0 on success, 1 on an argument error. */
int orc_causal_masked(const orc_params* p, const double* q, const double* k, const double* v,
                      const double* decay, const double* beta, const unsigned char* mask,
                      const double* S0, const double* Z0, double* y, double* S_out, double* Z_out)
{
    if (orc_check(p, 1, decay, beta)) return 1;
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.p = p; J.q = q; J.k = k; J.v = v; J.decay = decay; J.beta = beta; J.mask = mask;
    J.S0 = S0; J.Z0 = Z0; J.y = y; J.S_out = S_out; J.Z_out = Z_out; J.causal = 1;
    return orc_run(&J);
}

int orc_causal(const orc_params* p, const double* q, const double* k, const double* v,
               const double* decay, const double* beta, const double* S0, const double* Z0,
               double* y, double* S_out, double* Z_out)
{
    return orc_causal_masked(p, q, k, v, decay, beta, NULL, S0, Z0, y, S_out, Z_out);
}

/* Non-causal pass: global state over all (valid) positions, no state in or
 * out.  mask (B,T) as for orc_causal_masked, NULL = all valid. */
int orc_noncausal_masked(const orc_params* p, const double* q, const double* k, const double* v,
                         const unsigned char* mask, double* y)
{
    if (orc_check(p, 0, NULL, NULL)) return 1;
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.p = p; J.q = q; J.k = k; J.v = v; J.mask = mask; J.y = y; J.causal = 0;
    return orc_run(&J);
}

int orc_noncausal(const orc_params* p, const double* q, const double* k, const double* v, double* y)
{
    return orc_noncausal_masked(p, q, k, v, NULL, y);
}
