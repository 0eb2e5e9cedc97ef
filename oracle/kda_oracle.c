/*
 * Kimi Delta Attention (KDA) reference oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU evaluation of the gated delta-rule recurrence,
 * one token at a time.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code; the CUDA library never
 * calls it and shares no code with it.
 *
 * What it follows:
 *   - Lecture transcript "Inside Kimi K3: Architecture of an Open Frontier
 *     Model", paragraph on the sequence direction: every token rewrites a
 *     state of fixed shape in two stages -- the previous state is first
 *     shrunk channel by channel by a diagonal decay (the forget gate alpha),
 *     then a correction scaled by beta and built from k and v is added.  The
 *     log of the decay may not go below -5.
 *   - meridianbulletin.com article on Kimi K3, section "Handling One Million
 *     Tokens with a Fixed-Size State Matrix": beta is the overwrite strength,
 *     alpha the forgetting factor, and alpha is kept inside [e^-5, 1].
 *   - Written as one equation (the plainest reading of both), per head:
 *         S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *         o_t = S_t^T q_t
 *     with S of shape dk x dv and alpha_t = exp(clamp(log_alpha_t, -5, 0)),
 *     one value per key channel.
 *
 * The step is evaluated in the algebraically equal form
 *         S' = Diag(alpha_t) S_{t-1}
 *         u  = beta_t (v_t - S'^T k_t)
 *         S_t = S' + k_t u^T
 *         o_t = S_t^T q_t           (the updated state is read)
 * which is the expansion of (I - beta k k^T) S' + beta k v^T.
 *
 * Layouts (row-major, innermost last):
 *   q, k       [total_T, H, dk]        v, out   [total_T, H, dv]
 *   log_alpha  [total_T, H, dk]        beta     [total_T, H]
 *   S0, S_final [n_seqs, H, dk, dv]    cu_seqlens int64 [n_seqs + 1]
 * Sequence n owns tokens cu_seqlens[n] .. cu_seqlens[n+1]-1.
 *
 * Input encodings: ORACLE_IN_F64 -- every input is an fp64 array;
 * ORACLE_IN_BF16 -- q, k, v are bfloat16 bit patterns (uint16), log_alpha,
 * beta and S0 are fp32.  Every input value is widened exactly to fp64 before
 * use; all arithmetic is fp64.  Outputs are always fp64.
 *
 * Parallelism: independent (sequence, head) chains are spread over POSIX
 * threads; each chain is evaluated sequentially, so the result does not
 * depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_IN_F64 = 0, ORACLE_IN_BF16 = 1 };

typedef struct {
    const void *q, *k, *v, *log_alpha, *beta, *S0;
    const int64_t *cu_seqlens;
    int64_t n_seqs, H, dk, dv;
    int64_t head_begin, head_end; /* heads evaluated: [head_begin, head_end) */
    int in_kind;
    double *out;     /* [total_T, head_end - head_begin, dv] */
    double *S_final; /* [n_seqs, head_end - head_begin, dk, dv], nullable */
    /* work distribution */
    int64_t n_chains;
    int64_t next_chain;
    pthread_mutex_t lock;
    int error;
} oracle_job;

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_f64(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Element i of a q/k/v array. */
static double load_qkv(const oracle_job *job, const void *p, int64_t i)
{
    if (job->in_kind == ORACLE_IN_BF16)
        return bf16_bits_to_f64(((const uint16_t *)p)[i]);
    return ((const double *)p)[i];
}

/* Element i of a log_alpha / beta / S0 array. */
static double load_gate(const oracle_job *job, const void *p, int64_t i)
{
    if (job->in_kind == ORACLE_IN_BF16)
        return (double)((const float *)p)[i];
    return ((const double *)p)[i];
}

/* Scratch vectors of one chain: the decoded token and the update vector. */
typedef struct {
    double *S;     /* dk x dv state, row c = key channel */
    double *alpha; /* dk */
    double *q, *k; /* dk */
    double *v, *u; /* dv */
} chain_scratch;

/* One (sequence, head) chain, token by token. */
static void run_chain(const oracle_job *job, int64_t n, int64_t h,
                      const chain_scratch *w)
{
    const int64_t H = job->H, dk = job->dk, dv = job->dv;
    const int64_t nh = job->head_end - job->head_begin;
    const int64_t hs = h - job->head_begin; /* head index in the outputs */
    double *S = w->S;

    /* initial state: S0, or zero when no S0 is given */
    for (int64_t c = 0; c < dk; ++c)
        for (int64_t j = 0; j < dv; ++j)
            S[c * dv + j] = job->S0
                ? load_gate(job, job->S0, ((n * H + h) * dk + c) * dv + j)
                : 0.0;

    for (int64_t t = job->cu_seqlens[n]; t < job->cu_seqlens[n + 1]; ++t) {
        const int64_t qk_base = (t * H + h) * dk;
        const int64_t v_base = (t * H + h) * dv;

        /* decode the token; forget gate alpha = exp(clamp(log_alpha, -5, 0)) */
        for (int64_t c = 0; c < dk; ++c) {
            double la = load_gate(job, job->log_alpha, qk_base + c);
            if (la < -5.0) la = -5.0;
            if (la > 0.0) la = 0.0;
            w->alpha[c] = exp(la);
            w->q[c] = load_qkv(job, job->q, qk_base + c);
            w->k[c] = load_qkv(job, job->k, qk_base + c);
        }
        for (int64_t j = 0; j < dv; ++j)
            w->v[j] = load_qkv(job, job->v, v_base + j);
        const double b = load_gate(job, job->beta, t * H + h);

        /* S' = Diag(alpha) S */
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < dv; ++j)
                S[c * dv + j] *= w->alpha[c];
        /* u = beta (v - S'^T k) */
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int64_t c = 0; c < dk; ++c)
                acc += S[c * dv + j] * w->k[c];
            w->u[j] = b * (w->v[j] - acc);
        }
        /* S = S' + k u^T */
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < dv; ++j)
                S[c * dv + j] += w->k[c] * w->u[j];
        /* o = S^T q, reading the updated state */
        double *o = job->out + (t * nh + hs) * dv;
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int64_t c = 0; c < dk; ++c)
                acc += S[c * dv + j] * w->q[c];
            o[j] = acc;
        }
    }

    if (job->S_final)
        memcpy(job->S_final + (n * nh + hs) * dk * dv, S,
               (size_t)(dk * dv) * sizeof(double));
}

static void *worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const int64_t nh = job->head_end - job->head_begin;
    const size_t dk = (size_t)job->dk, dv = (size_t)job->dv;
    double *mem = malloc((dk * dv + 3 * dk + 2 * dv) * sizeof(double));
    if (!mem) {
        pthread_mutex_lock(&job->lock);
        job->error = 1;
        pthread_mutex_unlock(&job->lock);
        return NULL;
    }
    chain_scratch w;
    w.S = mem;
    w.alpha = w.S + dk * dv;
    w.q = w.alpha + dk;
    w.k = w.q + dk;
    w.v = w.k + dk;
    w.u = w.v + dv;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t chain = job->next_chain++;
        pthread_mutex_unlock(&job->lock);
        if (chain >= job->n_chains) break;
        int64_t n = chain / nh;
        int64_t h = job->head_begin + chain % nh;
        run_chain(job, n, h, &w);
    }
    free(mem);
    return NULL;
}

/*
 * Evaluate the recurrence for every sequence and the heads
 * [head_begin, head_end).  Returns 0 on success, -1 on a bad argument,
 * -2 when memory or threads cannot be obtained.
 */
int kda_oracle_forward(const void *q, const void *k, const void *v,
                       const void *log_alpha, const void *beta, const void *S0,
                       const int64_t *cu_seqlens, int64_t n_seqs, int64_t H,
                       int64_t dk, int64_t dv, int64_t head_begin,
                       int64_t head_end, int in_kind, double *out,
                       double *S_final, int n_threads)
{
    if (!q || !k || !v || !log_alpha || !beta || !cu_seqlens || !out)
        return -1;
    if (n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (head_begin < 0 || head_end > H || head_begin >= head_end) return -1;
    if (in_kind != ORACLE_IN_F64 && in_kind != ORACLE_IN_BF16) return -1;
    if (cu_seqlens[0] != 0) return -1;
    for (int64_t n = 0; n < n_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;

    oracle_job job;
    memset(&job, 0, sizeof job);
    job.q = q; job.k = k; job.v = v;
    job.log_alpha = log_alpha; job.beta = beta; job.S0 = S0;
    job.cu_seqlens = cu_seqlens;
    job.n_seqs = n_seqs; job.H = H; job.dk = dk; job.dv = dv;
    job.head_begin = head_begin; job.head_end = head_end;
    job.in_kind = in_kind;
    job.out = out; job.S_final = S_final;
    job.n_chains = n_seqs * (head_end - head_begin);
    job.next_chain = 0;
    pthread_mutex_init(&job.lock, NULL);

    if (n_threads < 1) n_threads = 1;
    if (n_threads > job.n_chains) n_threads = (int)(job.n_chains > 0 ? job.n_chains : 1);
    pthread_t *tid = malloc((size_t)n_threads * sizeof(pthread_t));
    if (!tid) { pthread_mutex_destroy(&job.lock); return -2; }
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&tid[i], NULL, worker, &job) != 0) break;
        ++started;
    }
    if (started == 0) worker(&job); /* no thread could start: run inline */
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&job.lock);
    return job.error ? -2 : 0;
}
