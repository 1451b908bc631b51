/*
 * KDA forward oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 token-by-token evaluation of the Kimi Delta Attention
 * forward pass.  Only the tests, the smoke check and the benchmark's CPU
 * baseline use it; the CUDA library never links, loads or calls it, and this
 * file shares no code with it.
 *
 * What it computes (per sequence n and head h, state S in R^{K x V}, K = V = 128):
 *
 *   q^ = q / sqrt(sum q^2 + 1e-6),  k^ = k / sqrt(sum k^2 + 1e-6)     (L2 norm in the kernel)
 *   b  = sigmoid(beta_logit)                                        (beta sigmoid in the kernel)
 *   a_c = lower_bound * sigmoid(exp(A_log[h]) * (g_c + dt_bias[h][c]))  (gate, c = 0..127)
 *   S' = Diag(exp(a)) S                                             (per-key-channel decay)
 *   S  = S' + k^ (b (v - S'^T k^))^T                                (delta-rule write)
 *   o  = scale * S^T q^                                             (read-out after the write)
 *
 * Sources: the FlashKDA README mirror (ai-feeds.com, "FlashKDA"), section
 * "内核 API" (argument table: shapes, dtypes, beta logits with the sigmoid applied
 * inside, scale, A_log / dt_bias / lower_bound, states [N,H,V,K], cu_seqlens rules)
 * and section "将 FlashKDA 用作 FLA 后端" (q/k L2 norm, beta sigmoid and the gate
 * computed inside the kernel, transposed [V,K] state layout); the guancyxx.cn
 * FlashKDA article, section 一 (recurrent state S of shape [K,V], gated decay) and
 * section 2.2 (the chunk-wise delta-rule recurrence that the chunked kernels
 * evaluate).  The pages do not print the gate activation; the form above is the
 * reading this project adopts: it is bounded in (lower_bound, 0) as a lower bound
 * requires.  The pages also print no L2-norm epsilon; 1e-6 is added to the sum of
 * squares.
 *
 * Precision: q, k, v, g, beta arrive as bf16 bit patterns and are widened
 * exactly; all arithmetic is IEEE fp64 with libm's exp and sqrt.  States and
 * outputs are fp64; rounding to a storage type is left to the caller.
 *
 * Layouts (row-major): q, k, v, g, out [rows, H, 128]; beta [rows, H];
 * A_log [H]; dt_bias [H, 128]; states [N, H, V, K], state[n][h][v][k] = S[k][v].
 * Without cu_seqlens, rows = N * T and sequence n is rows [n*T, (n+1)*T);
 * with cu_seqlens, rows = T and sequence n is rows [cu[n], cu[n+1]).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KDA_D 128

static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

typedef struct {
    const uint16_t *q, *k, *v, *g, *beta;
    double scale;
    double *out;
    const float *A_log, *dt_bias;
    double lower_bound;
    const double *initial_state;
    double *final_state;
    const int64_t *cu_seqlens;
    int N, H;
    int64_t T;
    int64_t next_pair; /* work counter shared by the threads */
} kda_oracle_job;

/* Evaluate one (sequence, head) pair from its first token to its last. */
static void oracle_pair(const kda_oracle_job *job, int n, int h, double *S)
{
    const int H = job->H;
    const int64_t bos = job->cu_seqlens ? job->cu_seqlens[n] : (int64_t)n * job->T;
    const int64_t eos = job->cu_seqlens ? job->cu_seqlens[n + 1] : (int64_t)(n + 1) * job->T;
    double qh[KDA_D], kh[KDA_D], alpha[KDA_D], u[KDA_D];

    /* S[kk][vv] from state[n][h][vv][kk] */
    for (int kk = 0; kk < KDA_D; ++kk)
        for (int vv = 0; vv < KDA_D; ++vv)
            S[kk * KDA_D + vv] = job->initial_state
                ? job->initial_state[(((int64_t)n * H + h) * KDA_D + vv) * KDA_D + kk]
                : 0.0;

    const double ea = exp((double)job->A_log[h]);
    const float *dtb = job->dt_bias + (int64_t)h * KDA_D;

    for (int64_t t = bos; t < eos; ++t) {
        const int64_t row = (t * H + h) * KDA_D;
        double sq = 0.0, sk = 0.0;
        for (int c = 0; c < KDA_D; ++c) {
            qh[c] = bf16_to_f64(job->q[row + c]);
            kh[c] = bf16_to_f64(job->k[row + c]);
            sq += qh[c] * qh[c];
            sk += kh[c] * kh[c];
        }
        const double rq = 1.0 / sqrt(sq + 1e-6), rk = 1.0 / sqrt(sk + 1e-6);
        for (int c = 0; c < KDA_D; ++c) {
            qh[c] *= rq;
            kh[c] *= rk;
        }
        const double b = sigmoid(bf16_to_f64(job->beta[t * H + h]));
        for (int c = 0; c < KDA_D; ++c) {
            const double z = ea * (bf16_to_f64(job->g[row + c]) + (double)dtb[c]);
            alpha[c] = exp(job->lower_bound * sigmoid(z));
        }
        /* S' = Diag(alpha) S */
        for (int kk = 0; kk < KDA_D; ++kk)
            for (int vv = 0; vv < KDA_D; ++vv)
                S[kk * KDA_D + vv] *= alpha[kk];
        /* u = b (v - S'^T k^) */
        for (int vv = 0; vv < KDA_D; ++vv) {
            double p = 0.0;
            for (int kk = 0; kk < KDA_D; ++kk)
                p += S[kk * KDA_D + vv] * kh[kk];
            u[vv] = b * (bf16_to_f64(job->v[row + vv]) - p);
        }
        /* S = S' + k^ u^T */
        for (int kk = 0; kk < KDA_D; ++kk)
            for (int vv = 0; vv < KDA_D; ++vv)
                S[kk * KDA_D + vv] += kh[kk] * u[vv];
        /* o = scale S^T q^ */
        for (int vv = 0; vv < KDA_D; ++vv) {
            double o = 0.0;
            for (int kk = 0; kk < KDA_D; ++kk)
                o += S[kk * KDA_D + vv] * qh[kk];
            job->out[row + vv] = job->scale * o;
        }
    }

    if (job->final_state)
        for (int kk = 0; kk < KDA_D; ++kk)
            for (int vv = 0; vv < KDA_D; ++vv)
                job->final_state[(((int64_t)n * H + h) * KDA_D + vv) * KDA_D + kk] = S[kk * KDA_D + vv];
}

static void *oracle_worker(void *arg)
{
    kda_oracle_job *job = (kda_oracle_job *)arg;
    double *S = (double *)malloc(sizeof(double) * KDA_D * KDA_D);
    if (!S)
        return (void *)1;
    const int64_t pairs = (int64_t)job->N * job->H;
    for (;;) {
        const int64_t p = __atomic_fetch_add(&job->next_pair, 1, __ATOMIC_RELAXED);
        if (p >= pairs)
            break;
        oracle_pair(job, (int)(p / job->H), (int)(p % job->H), S);
    }
    free(S);
    return NULL;
}

/*
 * Returns 0 on success; -1 for invalid arguments; -2 when a thread could not be
 * started or could not allocate its state.  All pointers are host pointers.
 * T is the per-sequence length without cu_seqlens and the total length with it.
 * initial_state and final_state may be NULL (zero initial state / no output).
 */
int kda_oracle_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *g,
                   const uint16_t *beta, double scale, double *out, const float *A_log,
                   const float *dt_bias, double lower_bound, const double *initial_state,
                   double *final_state, const int64_t *cu_seqlens, int N, int64_t T, int H,
                   int nthreads)
{
    if (!q || !k || !v || !g || !beta || !out || !A_log || !dt_bias || N < 1 || H < 1 || T < 0)
        return -1;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0 || cu_seqlens[N] != T)
            return -1;
        for (int n = 0; n < N; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n])
                return -1;
    }
    if (nthreads < 1)
        nthreads = 1;
    if ((int64_t)nthreads > (int64_t)N * H)
        nthreads = (int)((int64_t)N * H);

    kda_oracle_job job = {q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                          initial_state, final_state, cu_seqlens, N, H, T, 0};
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!tids)
        return -2;
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&tids[i], NULL, oracle_worker, &job) != 0) {
            rc = -2;
            break;
        }
        ++started;
    }
    if (started == 0)
        rc = -2;
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tids[i], &ret);
        if (ret)
            rc = -2;
    }
    free(tids);
    return rc;
}
