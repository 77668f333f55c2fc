/*
 * gdr_oracle.c -- plain float64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers. The product path (the CUDA library and
 * its Python binding) never loads, links or calls this file, and this file
 * shares no code, header, table or constant with it.
 *
 * What it computes, token by token, for every (sequence, head):
 *
 *   "Linear attention" (arsalanzafar.ai), section "How it works", Eqs. (1)-(4),
 *   with the state stored keys x values (S is d_k x d_v, d_v contiguous):
 *     (1)  S'_t    = alpha_t S_{t-1}
 *     (2)  vhat_t  = S'_t^T k_t
 *     (3)  S_t     = S'_t + beta_t k_t (v_t - vhat_t)^T
 *     (4)  o_t     = S_t^T q_t
 *   alpha_t = exp(log_alpha_t). The state is updated first and read second
 *   ("How linear attention works: a small memory matrix and the gated delta
 *   rule", section "Writing a key-value association": update first, then read).
 *   No score scale and no normalisation of q or k: the caller passes the
 *   vectors it wants used.
 *
 *   With `per_channel` set, alpha_t is a d_k vector: each key channel (row i of
 *   S) has its own rate, S'_t = diag(alpha_t) S_{t-1} ("Attention as Matrix
 *   Algebra: From Softmax to the Delta Rule", section 10 "Where this goes next":
 *   Kimi Delta Attention gives each feature channel its own rate). The other
 *   steps are unchanged.
 *
 *   With `additive` set, step (2)-(3) is replaced by the decayed additive write
 *   S_t = alpha_t S_{t-1} + beta_t k_t v_t^T ("From KV Cache to a State Matrix:
 *   Linear Attention and DeltaNet", section "From attention weights to a state
 *   matrix", the decay-gate form, and section "Associating keys and values",
 *   the gradient step on the dot-product loss with write strength beta_t).
 *   It exists only so that tests can check the additive special case.
 *
 * Everything is float64; inputs are the exact values the GPU receives, widened.
 * Work items (sequence, head) are independent; they are spread over POSIX
 * threads. Each item runs the plain token loop above, nothing is blocked,
 * fused or reordered.
 *
 * Layouts (all row-major, contiguous):
 *   q, k        [total_tokens, H, dk]
 *   v, o        [total_tokens, H, dv]
 *   log_alpha   [total_tokens, H], or [total_tokens, H, dk] with per_channel
 *   beta        [total_tokens, H]
 *   S0, S_final [num_seqs, H, dk, dv]     (S0 may be NULL: zero state)
 *   cu_seqlens  [num_seqs + 1] int64 offsets into the token axis, or NULL
 *               for num_seqs equal sequences of total_tokens / num_seqs tokens.
 * Returns 0 on success, -1 on an invalid argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* One token of Eqs. (1)-(4) on the state S (dk x dv). log_alpha points at the token's
 * one rate, or at its dk rates with per_channel. `scratch` holds dv doubles. */
static void oracle_token(double *S, int64_t dk, int64_t dv, const double *q, const double *k,
                         const double *v, const double *log_alpha, int per_channel, double beta,
                         int additive, double *o, double *scratch)
{
    int64_t i, j;

    /* (1) decay: row i (key channel i) by alpha_t, or by its own alpha_t[i] */
    for (i = 0; i < dk; ++i) {
        const double alpha = exp(log_alpha[per_channel ? i : 0]);
        for (j = 0; j < dv; ++j)
            S[i * dv + j] *= alpha;
    }

    if (additive) {
        /* decayed additive write: S += beta k v^T */
        for (i = 0; i < dk; ++i)
            for (j = 0; j < dv; ++j)
                S[i * dv + j] += beta * k[i] * v[j];
    } else {
        /* (2) vhat = S'^T k : vhat_j = sum_i S'_ij k_i */
        double *vhat = scratch;
        for (j = 0; j < dv; ++j)
            vhat[j] = 0.0;
        for (i = 0; i < dk; ++i)
            for (j = 0; j < dv; ++j)
                vhat[j] += S[i * dv + j] * k[i];
        /* (3) S = S' + beta k (v - vhat)^T */
        for (i = 0; i < dk; ++i)
            for (j = 0; j < dv; ++j)
                S[i * dv + j] += beta * k[i] * (v[j] - vhat[j]);
    }

    /* (4) o = S^T q : o_j = sum_i S_ij q_i */
    for (j = 0; j < dv; ++j)
        o[j] = 0.0;
    for (i = 0; i < dk; ++i)
        for (j = 0; j < dv; ++j)
            o[j] += S[i * dv + j] * q[i];
}

typedef struct {
    const double *q, *k, *v, *log_alpha, *beta, *S0;
    const int64_t *cu;      /* may be NULL */
    int64_t num_seqs, total_tokens, H, dk, dv, seq_len;
    int additive, per_channel;
    double *o, *S_final;
    int64_t first_item, item_stride;
    int status;
} oracle_job;

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const int64_t H = job->H, dk = job->dk, dv = job->dv;
    double *scratch = (double *)malloc((size_t)dv * sizeof(double));
    if (!scratch) {
        job->status = -2;
        return NULL;
    }
    for (int64_t item = job->first_item; item < job->num_seqs * H; item += job->item_stride) {
        const int64_t n = item / H, h = item % H;
        const int64_t t0 = job->cu ? job->cu[n] : n * job->seq_len;
        const int64_t t1 = job->cu ? job->cu[n + 1] : (n + 1) * job->seq_len;
        double *S = job->S_final + (n * H + h) * dk * dv;
        if (job->S0)
            memmove(S, job->S0 + (n * H + h) * dk * dv, (size_t)(dk * dv) * sizeof(double));
        else
            memset(S, 0, (size_t)(dk * dv) * sizeof(double));
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t th = t * H + h;
            oracle_token(S, dk, dv, job->q + th * dk, job->k + th * dk, job->v + th * dv,
                         job->log_alpha + th * (job->per_channel ? dk : 1), job->per_channel,
                         job->beta[th], job->additive, job->o + th * dv, scratch);
        }
    }
    free(scratch);
    return NULL;
}

static int run_jobs(oracle_job *proto, int nthreads)
{
    const int64_t items = proto->num_seqs * proto->H;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > items)
        nthreads = items > 0 ? (int)items : 1;
    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int status = 0;
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = *proto;
        jobs[i].first_item = i;
        jobs[i].item_stride = nthreads;
        jobs[i].status = 0;
    }
    if (nthreads == 1) {
        oracle_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int i = 0; i < nthreads; ++i) {
            if (pthread_create(&tids[i], NULL, oracle_worker, &jobs[i]) != 0) {
                /* run it on this thread instead */
                oracle_worker(&jobs[i]);
                tids[i] = 0;
            } else {
                ++started;
            }
        }
        for (int i = 0; i < nthreads; ++i)
            if (tids[i])
                pthread_join(tids[i], NULL);
        (void)started;
    }
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].status)
            status = jobs[i].status;
    free(jobs);
    free(tids);
    return status;
}

int gdr_oracle_forward(const double *q, const double *k, const double *v,
                       const double *log_alpha, const double *beta, const double *S0,
                       const int64_t *cu_seqlens, int64_t num_seqs, int64_t total_tokens,
                       int64_t H, int64_t dk, int64_t dv, int additive, int per_channel,
                       int nthreads, double *o, double *S_final)
{
    if (num_seqs < 0 || total_tokens < 0 || H <= 0 || dk <= 0 || dv <= 0 || !S_final)
        return -1;
    if (total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !o))
        return -1;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != total_tokens)
            return -1;
        for (int64_t n = 0; n < num_seqs; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n])
                return -1;
    } else if (num_seqs > 0 && total_tokens % num_seqs != 0) {
        return -1;
    }
    if (num_seqs == 0)
        return 0;
    oracle_job proto;
    memset(&proto, 0, sizeof(proto));
    proto.q = q;
    proto.k = k;
    proto.v = v;
    proto.log_alpha = log_alpha;
    proto.beta = beta;
    proto.S0 = S0;
    proto.cu = cu_seqlens;
    proto.num_seqs = num_seqs;
    proto.total_tokens = total_tokens;
    proto.H = H;
    proto.dk = dk;
    proto.dv = dv;
    proto.seq_len = cu_seqlens ? 0 : total_tokens / num_seqs;
    proto.additive = additive;
    proto.per_channel = per_channel;
    proto.o = o;
    proto.S_final = S_final;
    return run_jobs(&proto, nthreads);
}

/*
 * One decode step: one token per sequence, the state updated in place.
 * Layouts: q, k [N, H, dk]; v, o [N, H, dv]; log_alpha [N, H] (or [N, H, dk] with
 * per_channel), beta [N, H]; S [N, H, dk, dv]. It is gdr_oracle_forward with one
 * token per sequence and S0 = S_final = S.
 */
int gdr_oracle_decode(const double *q, const double *k, const double *v, const double *log_alpha,
                      const double *beta, double *S, double *o, int64_t N, int64_t H, int64_t dk,
                      int64_t dv, int per_channel, int nthreads)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0)
        return -1;
    if (N == 0)
        return 0;
    if (!q || !k || !v || !log_alpha || !beta || !S || !o)
        return -1;
    return gdr_oracle_forward(q, k, v, log_alpha, beta, S, NULL, N, N, H, dk, dv, 0, per_channel,
                              nthreads, o, S);
}
