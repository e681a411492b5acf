/*
 * kda_oracle.c -- fp64 CPU oracle of the Kimi Delta Attention (KDA) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: it exists so that tests, the smoke check and the benchmark's CPU
 * baseline can compare the CUDA library against a plain, slow, obviously
 * correct restatement of what the method computes.  It shares no code, header
 * or constant with the CUDA sources.
 *
 * What it computes (one (sequence, head) unit at a time, token by token, in
 * double precision, no chunking, no reordering):
 *
 *   S            <- initial state of the unit (zero when none is given)
 *   for every token t of the sequence, in order:
 *     a_i        = exp(log_alpha[t,i])                      per key channel i
 *     St[i][j]   = a_i * S[i][j]                            decay the key rows
 *     p_j        = sum_i St[i][j] * k[t,i]                  prediction St^T k
 *     d_j        = beta[t] * (v[t,j] - p_j)                 scaled residual
 *     S[i][j]    = St[i][j] + k[t,i] * d_j                  delta-rule write
 *     o[t,j]     = sum_i S[i][j] * q[t,i] / sqrt(d_k)       read after the write
 *   final state of the unit = S
 *
 * Sources (web pages on Kimi K3 / Kimi Linear):
 *  - "Day 19, linear attention & KDA" (ai.air7.fun k3-course-30), section 3,
 *    the two update lines: first the per-channel decay of the state, then the
 *    delta correction of the decayed state with strength beta_t.
 *  - "K3 attention, three-piece set" (yeyulingfeng.com), KDA paragraphs: the
 *    (I - beta_t k_t k_t^T) factor (subtract what the old state holds along the
 *    new key, then write the new pair), and the per-channel gate Diag(alpha_t)
 *    with alpha_t a vector over the d_k key channels.
 *  - "From 124M to 2.8T" (ciyuanerhao.com), chapter 4 gate code: alpha has
 *    one value per key channel and scales the key rows of S = k^T u
 *    (alpha.unsqueeze(-1) * S); chapter 3 DeltaNet code: u = beta (v - k S),
 *    S = S + k^T u, then o = q S (the read uses the updated state).
 *  - The pages give no output scale; the library defines o with q scaled by
 *    1/sqrt(d_k), and so does this oracle.
 *
 * Matrix convention: S is d_k x d_v (row = key channel i, column = value
 * channel j), so the prediction is S^T k and the output is S^T q.
 *
 * Threads: units are independent, so they are spread over POSIX threads; each
 * unit is still computed strictly token by token.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    /* token-major tensors: [total_tokens, H, d] */
    const double *q, *k, *v, *log_alpha, *beta;
    const int64_t *cu_seqlens; /* [num_seqs + 1] */
    int64_t num_seqs, H, dk, dv;
    const double *init_state; /* [num_seqs, H, dk, dv] or NULL */
    double *o;                /* [total_tokens, H, dv] (may be NULL) */
    double *final_state;      /* [num_seqs, H, dk, dv] */
    int64_t next_unit;        /* shared work counter */
    pthread_mutex_t lock;
} prefill_job;

/* One token of the recurrence on one unit's state S (dk x dv, row-major).
 * scratch must hold dv doubles.  Writes the output row when o_row != NULL. */
static void kda_token(double *S, int64_t dk, int64_t dv, const double *q, const double *k,
                      const double *v, const double *log_alpha, double beta, double *o_row,
                      double *scratch)
{
    const double scale = 1.0 / sqrt((double)dk);
    double *d = scratch;
    /* decay: row i of S is multiplied by alpha_i */
    for (int64_t i = 0; i < dk; ++i) {
        const double a = exp(log_alpha[i]);
        for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a;
    }
    /* residual of the prediction St^T k against v, scaled by beta */
    for (int64_t j = 0; j < dv; ++j) {
        double p = 0.0;
        for (int64_t i = 0; i < dk; ++i) p += S[i * dv + j] * k[i];
        d[j] = beta * (v[j] - p);
    }
    /* write: S = St + k d^T */
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += k[i] * d[j];
    /* read from the updated state */
    if (o_row) {
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * q[i];
            o_row[j] = acc * scale;
        }
    }
}

static void prefill_unit(prefill_job *J, int64_t unit, double *S, double *scratch)
{
    const int64_t n = unit / J->H, h = unit % J->H;
    const int64_t H = J->H, dk = J->dk, dv = J->dv;
    const int64_t t0 = J->cu_seqlens[n], t1 = J->cu_seqlens[n + 1];
    const int64_t state_off = (n * H + h) * dk * dv;
    if (J->init_state)
        memcpy(S, J->init_state + state_off, (size_t)(dk * dv) * sizeof(double));
    else
        memset(S, 0, (size_t)(dk * dv) * sizeof(double));
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t row = t * H + h;
        kda_token(S, dk, dv, J->q + row * dk, J->k + row * dk, J->v + row * dv,
                  J->log_alpha + row * dk, J->beta[row], J->o ? J->o + row * dv : NULL, scratch);
    }
    memcpy(J->final_state + state_off, S, (size_t)(dk * dv) * sizeof(double));
}

static void *prefill_worker(void *arg)
{
    prefill_job *J = (prefill_job *)arg;
    double *S = (double *)malloc((size_t)(J->dk * J->dv + J->dv) * sizeof(double));
    if (!S) return (void *)1;
    const int64_t units = J->num_seqs * J->H;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= units) break;
        prefill_unit(J, u, S, S + J->dk * J->dv);
    }
    free(S);
    return NULL;
}

static int resolve_threads(int nthreads, int64_t units)
{
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > units) nthreads = (int)(units > 0 ? units : 1);
    if (nthreads > 256) nthreads = 256;
    return nthreads;
}

/* Returns the number of threads used, or -1 on an allocation/thread failure. */
int kda_oracle_prefill(const double *q, const double *k, const double *v, const double *log_alpha,
                       const double *beta, const int64_t *cu_seqlens, int64_t num_seqs, int64_t H,
                       int64_t dk, int64_t dv, const double *init_state, double *o,
                       double *final_state, int nthreads)
{
    prefill_job J;
    J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha; J.beta = beta;
    J.cu_seqlens = cu_seqlens; J.num_seqs = num_seqs; J.H = H; J.dk = dk; J.dv = dv;
    J.init_state = init_state; J.o = o; J.final_state = final_state; J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);
    const int64_t units = num_seqs * H;
    const int nt = resolve_threads(nthreads, units);
    pthread_t tid[256];
    int started = 0, failed = 0;
    for (int i = 0; i < nt; ++i) {
        if (pthread_create(&tid[i], NULL, prefill_worker, &J) != 0) { failed = 1; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tid[i], &ret);
        if (ret) failed = 1;
    }
    pthread_mutex_destroy(&J.lock);
    if (started == 0) return -1;
    return failed ? -1 : started;
}

typedef struct {
    const double *q, *k, *v, *log_alpha, *beta;
    int64_t B, H, dk, dv;
    double *state, *o;
    int64_t next_unit;
    pthread_mutex_t lock;
} decode_job;

static void *decode_worker(void *arg)
{
    decode_job *J = (decode_job *)arg;
    double *scratch = (double *)malloc((size_t)J->dv * sizeof(double));
    if (!scratch) return (void *)1;
    const int64_t units = J->B * J->H;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= units) break;
        kda_token(J->state + u * J->dk * J->dv, J->dk, J->dv, J->q + u * J->dk, J->k + u * J->dk,
                  J->v + u * J->dv, J->log_alpha + u * J->dk, J->beta[u], J->o + u * J->dv,
                  scratch);
    }
    free(scratch);
    return NULL;
}

/* One decode step for B sequences x H heads: the loop body above, applied once
 * to the caller's state [B, H, dk, dv] in place.  q,k,log_alpha: [B,H,dk];
 * v, o: [B,H,dv]; beta: [B,H].  Returns the thread count or -1. */
int kda_oracle_decode_step(const double *q, const double *k, const double *v,
                           const double *log_alpha, const double *beta, int64_t B, int64_t H,
                           int64_t dk, int64_t dv, double *state, double *o, int nthreads)
{
    decode_job J;
    J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha; J.beta = beta;
    J.B = B; J.H = H; J.dk = dk; J.dv = dv; J.state = state; J.o = o; J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);
    const int nt = resolve_threads(nthreads, B * H);
    pthread_t tid[256];
    int started = 0, failed = 0;
    for (int i = 0; i < nt; ++i) {
        if (pthread_create(&tid[i], NULL, decode_worker, &J) != 0) { failed = 1; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tid[i], &ret);
        if (ret) failed = 1;
    }
    pthread_mutex_destroy(&J.lock);
    if (started == 0) return -1;
    return failed ? -1 : started;
}
