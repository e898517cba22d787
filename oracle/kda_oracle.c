/*
 * kda_oracle.c -- fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline arm may load this library.  The product path (the
 * CUDA library under gated_delta_rule_46_gb300/) never calls it and shares no
 * code, header, table or helper with it.
 *
 * What it computes, and where that is defined:
 *
 *  - The bounded gate.  "Kimi K3 internals analysis" (molayo1419.me), section
 *    "Sequence mixing": g = g_min * sigmoid(exp(A) * z), alpha = exp(g),
 *    g_min = -5.  The decay is per key channel (the channel-wise retention
 *    factor of the same section).
 *
 *  - The recurrence.  Same section: KDA replaces the length-dependent KV cache
 *    by a fixed-size state written by the delta rule, and the channel-wise
 *    retention factor decides how much of the old state survives *before* the
 *    current key/value pair is written.  The page gives this in prose only; the
 *    formula used here is the plain reading of it:
 *        S'  = Diag(alpha_t) S_{t-1}
 *        u_t = beta_t (v_t - S'^T k_t)
 *        S_t = S' + k_t u_t^T
 *        o_t = S_t^T q_t
 *    with S of shape [dk, dv] (rows = key channels), no 1/sqrt(dk) scale on q,
 *    and beta_t a scalar per (token, head) already passed through its sigmoid.
 *
 * It is written token by token in double precision with no blocking, no
 * chunking and no reordering: one (sequence, head) chain per work item, chains
 * spread over POSIX threads.  Inputs arrive as float32 (bf16 inputs upcast to
 * float32 exactly by the caller); every arithmetic step below is in double.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KDA_ORACLE_G_MIN (-5.0)

/* g = g_min * sigmoid(exp(A) * z); the sigmoid is 1 / (1 + exp(-x)). */
static double oracle_gate(double z, double A)
{
    double x = exp(A) * z;
    return KDA_ORACLE_G_MIN / (1.0 + exp(-x));
}

void kda_oracle_gate(const float *z, const float *A, double *g_out,
                     int64_t n_tokens, int H, int dk)
{
    for (int64_t t = 0; t < n_tokens; ++t)
        for (int h = 0; h < H; ++h)
            for (int c = 0; c < dk; ++c) {
                int64_t i = (t * H + h) * (int64_t)dk + c;
                g_out[i] = oracle_gate((double)z[i], (double)A[(int64_t)h * dk + c]);
            }
}

typedef struct {
    const float *q, *k, *v, *z, *A, *beta;
    const double *g_direct;      /* optional: log-decay given directly [T,H,dk] */
    const int64_t *cu_seqlens;   /* [num_seqs + 1] */
    int num_seqs, H, dk, dv;
    const double *initial_state; /* optional [num_seqs, H, dk, dv] */
    double *final_state;         /* optional [num_seqs, H, dk, dv] */
    double *out;                 /* [T, H, dv] */
    int64_t next_chain;          /* shared work counter */
    pthread_mutex_t lock;
} oracle_job;

/* One (sequence, head) chain, token by token. */
static void oracle_chain(oracle_job *job, int seq, int h, double *S, double *alpha,
                         double *kv, double *u)
{
    const int H = job->H, dk = job->dk, dv = job->dv;
    const int64_t bos = job->cu_seqlens[seq], eos = job->cu_seqlens[seq + 1];
    const int64_t sidx = ((int64_t)seq * H + h) * (int64_t)dk * dv;

    if (job->initial_state)
        memcpy(S, job->initial_state + sidx, sizeof(double) * (size_t)dk * dv);
    else
        memset(S, 0, sizeof(double) * (size_t)dk * dv);

    for (int64_t t = bos; t < eos; ++t) {
        const int64_t rk = (t * H + h) * (int64_t)dk; /* row of q, k, z, g */
        const int64_t rv = (t * H + h) * (int64_t)dv; /* row of v, o */
        const double b = (double)job->beta[t * H + h];

        /* channel-wise retention alpha = exp(g) */
        for (int c = 0; c < dk; ++c) {
            double g = job->g_direct ? job->g_direct[rk + c]
                                     : oracle_gate((double)job->z[rk + c],
                                                   (double)job->A[(int64_t)h * dk + c]);
            alpha[c] = exp(g);
        }
        /* S' = Diag(alpha) S : the old state decays before the write */
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j)
                S[(int64_t)c * dv + j] *= alpha[c];
        /* kv = S'^T k */
        for (int j = 0; j < dv; ++j) kv[j] = 0.0;
        for (int c = 0; c < dk; ++c) {
            double kc = (double)job->k[rk + c];
            for (int j = 0; j < dv; ++j) kv[j] += S[(int64_t)c * dv + j] * kc;
        }
        /* u = beta (v - S'^T k) */
        for (int j = 0; j < dv; ++j) u[j] = b * ((double)job->v[rv + j] - kv[j]);
        /* S = S' + k u^T */
        for (int c = 0; c < dk; ++c) {
            double kc = (double)job->k[rk + c];
            for (int j = 0; j < dv; ++j) S[(int64_t)c * dv + j] += kc * u[j];
        }
        /* o = S^T q */
        double *o = job->out + rv;
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (int c = 0; c < dk; ++c) {
            double qc = (double)job->q[rk + c];
            for (int j = 0; j < dv; ++j) o[j] += S[(int64_t)c * dv + j] * qc;
        }
    }
    if (job->final_state)
        memcpy(job->final_state + sidx, S, sizeof(double) * (size_t)dk * dv);
}

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const int dk = job->dk, dv = job->dv;
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *alpha = (double *)malloc(sizeof(double) * (size_t)dk);
    double *kv = (double *)malloc(sizeof(double) * (size_t)dv);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    const int64_t n_chains = (int64_t)job->num_seqs * job->H;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t w = job->next_chain++;
        pthread_mutex_unlock(&job->lock);
        if (w >= n_chains) break;
        oracle_chain(job, (int)(w / job->H), (int)(w % job->H), S, alpha, kv, u);
    }
    free(S); free(alpha); free(kv); free(u);
    return NULL;
}

/*
 * Runs every (sequence, head) chain of a packed variable-length batch.
 * Layouts (row-major, contiguous): q, k, z [T, H, dk]; v [T, H, dv];
 * beta [T, H]; A [H, dk]; states [num_seqs, H, dk, dv]; out [T, H, dv].
 * Either z (with A) or g_direct supplies the log-decay.  Returns 0 on success,
 * -1 on bad arguments.
 */
int kda_oracle_prefill(const float *q, const float *k, const float *v,
                       const float *z, const float *A, const double *g_direct,
                       const float *beta, const int64_t *cu_seqlens, int num_seqs,
                       int H, int dk, int dv, const double *initial_state,
                       double *final_state, double *out, int n_threads)
{
    if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !q || !k || !v || !beta ||
        !cu_seqlens || !out || (!g_direct && (!z || !A)))
        return -1;
    for (int i = 0; i < num_seqs; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return -1;
    oracle_job job;
    job.q = q; job.k = k; job.v = v; job.z = z; job.A = A; job.beta = beta;
    job.g_direct = g_direct; job.cu_seqlens = cu_seqlens; job.num_seqs = num_seqs;
    job.H = H; job.dk = dk; job.dv = dv; job.initial_state = initial_state;
    job.final_state = final_state; job.out = out; job.next_chain = 0;
    pthread_mutex_init(&job.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 1024) n_threads = 1024;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&tid[started], NULL, oracle_worker, &job) == 0) ++started;
    oracle_worker(&job);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&job.lock);
    return 0;
}

/*
 * One decode step for N sequences: every sequence contributes exactly one new
 * token, and the state [N, H, dk, dv] is read and overwritten.  This is the
 * same recurrence as above with length-1 sequences.
 */
int kda_oracle_decode_step(const float *q, const float *k, const float *v,
                           const float *z, const float *A, const float *beta,
                           double *state, double *out, int N, int H, int dk,
                           int dv, int n_threads)
{
    int64_t *cu = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N + 1));
    for (int i = 0; i <= N; ++i) cu[i] = i;
    size_t nstate = (size_t)N * H * dk * dv;
    double *tmp = (double *)malloc(sizeof(double) * nstate);
    int rc = kda_oracle_prefill(q, k, v, z, A, NULL, beta, cu, N, H, dk, dv, state,
                                tmp, out, n_threads);
    if (rc == 0) memcpy(state, tmp, sizeof(double) * nstate);
    free(tmp);
    free(cu);
    return rc;
}
