/*
 * gqa_oracle.c -- plain, slow fp64 CPU oracle for causal grouped-query
 * attention over a KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library.  It shares no code,
 * header or constant with the CUDA library it checks.
 *
 * What it computes ("第二章 Prefill：整层状态演化与 KV 建立", section 2.3,
 * the attention sub-layer, equations for g(h), S, A and O):
 *
 *   g(h)        = floor(h * H_kv / H_q)                (query head -> KV head)
 *   S[i, j]     = <q[i, h], K[j, g(h)]> / sqrt(d_h) + M[i, j]
 *   M[i, j]     = 0 if key j is visible to query i, else -inf
 *   A[i, j]     = exp(S[i, j] - m_i) / sum_{k: S[i,k] > -inf} exp(S[i, k] - m_i)
 *                 with m_i the largest finite score of row i
 *   O[i, h, :]  = sum_j A[i, j] * V[j, g(h), :]
 *
 * Visibility (section 2.2, the mask M; and "KV Cache 与 Prefill/Decode 推理
 * 路径", the incremental-prefill lesson): a query at absolute position p sees
 * the cached keys at positions 0..p -- the whole old prefix plus the lower
 * triangle of its own block.  A single-token decode query at position L-1 sees
 * all L cached keys.  Keys are therefore passed as the sequence's logical
 * cache K[0..L), V[0..L) in position order, and each query row carries its
 * absolute position.
 *
 * The scores are kept only for j <= p: the -inf entries of M contribute
 * exactly nothing to the max, the denominator or the sum, which is the
 * definition's "sum over finite scores".
 *
 * Sliding window ("KV Cache 与 Prefill/Decode 推理路径", the sliding-window
 * and ring-cache lesson: position t reads the most recent W positions, the
 * current one included): with a window W > 0 the visible keys are
 * max(0, p - W + 1) .. p.  W <= 0 means no window.
 *
 * Threads: rows (i, h) are independent; they are dealt round-robin to
 * threads.  Each row is computed by the same sequential loops whatever the
 * thread count, so results do not depend on it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int n_q, H_q, H_kv, d, L;
    int64_t window;           /* <= 0: none                                  */
    const double *q;          /* [n_q][H_q][d]  */
    const int64_t *qpos;      /* [n_q]           */
    const double *K, *V;      /* [L][H_kv][d]    */
    double *out;              /* [n_q][H_q][d]  */
    int tid, nthreads;
    int status;
} orc_job;

/* g(h) = floor(h * H_kv / H_q): section 2.3 of the prefill chapter. */
static int kv_head_of(int h, int H_q, int H_kv)
{
    return (int)(((int64_t)h * (int64_t)H_kv) / (int64_t)H_q);
}

static void attend_row(const orc_job *J, int i, int h, double *s, double *a)
{
    const int d = J->d;
    const int g = kv_head_of(h, J->H_q, J->H_kv);
    const double *qi = J->q + ((size_t)i * J->H_q + h) * d;
    double *o = J->out + ((size_t)i * J->H_q + h) * d;
    const int64_t p = J->qpos[i];
    const int64_t j0 = (J->window > 0 && p - J->window + 1 > 0) ? p - J->window + 1 : 0;
    const double root_d = sqrt((double)d);

    /* S row over the visible keys j0..p, and its largest finite entry. */
    double m = -INFINITY;
    for (int64_t j = j0; j <= p; ++j) {
        const double *kj = J->K + ((size_t)j * J->H_kv + g) * d;
        double dot = 0.0;
        for (int e = 0; e < d; ++e)
            dot += qi[e] * kj[e];
        s[j] = dot / root_d;
        if (s[j] > m)
            m = s[j];
    }
    /* Denominator over finite scores, then the row of A. */
    double den = 0.0;
    for (int64_t j = j0; j <= p; ++j)
        den += exp(s[j] - m);
    for (int64_t j = j0; j <= p; ++j)
        a[j] = exp(s[j] - m) / den;
    /* O = A V. */
    for (int e = 0; e < d; ++e)
        o[e] = 0.0;
    for (int64_t j = j0; j <= p; ++j) {
        const double *vj = J->V + ((size_t)j * J->H_kv + g) * d;
        for (int e = 0; e < d; ++e)
            o[e] += a[j] * vj[e];
    }
}

static void *worker(void *arg)
{
    orc_job *J = (orc_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->L > 0 ? J->L : 1));
    double *a = (double *)malloc(sizeof(double) * (size_t)(J->L > 0 ? J->L : 1));
    if (!s || !a) {
        J->status = -2;
        free(s);
        free(a);
        return NULL;
    }
    const int64_t rows = (int64_t)J->n_q * J->H_q;
    for (int64_t r = J->tid; r < rows; r += J->nthreads)
        attend_row(J, (int)(r / J->H_q), (int)(r % J->H_q), s, a);
    free(s);
    free(a);
    return NULL;
}

/*
 * Causal GQA attention for one sequence.
 * Returns 0, or -1 when a precondition fails (H_kv does not divide H_q, a query
 * position outside [0, L) -- such a row would have no visible key), or -2 on
 * allocation failure.  Rows with qpos < 0 are rejected too: padding rows are
 * the caller's business and never reach the oracle.
 */
int orc_attention_window(int n_q, int H_q, int H_kv, int d,
                         const double *q, const int64_t *qpos,
                         int L, const double *K, const double *V,
                         double *out, int nthreads, int64_t window)
{
    if (n_q < 0 || H_q <= 0 || H_kv <= 0 || d <= 0 || L < 0 || H_q % H_kv != 0)
        return -1;
    for (int i = 0; i < n_q; ++i)
        if (qpos[i] < 0 || qpos[i] >= L)
            return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;

    orc_job jobs[256];
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        orc_job J = {n_q, H_q, H_kv, d, L, window, q, qpos, K, V, out, t, nthreads, 0};
        jobs[t] = J;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0)
            break;
        started = t;
    }
    /* Rows of threads that failed to start run on this thread. */
    for (int t = started + 1; t < nthreads; ++t)
        worker(&jobs[t]);
    worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0)
            return jobs[t].status;
    return 0;
}

/* The same without a window. */
int orc_attention(int n_q, int H_q, int H_kv, int d,
                  const double *q, const int64_t *qpos,
                  int L, const double *K, const double *V,
                  double *out, int nthreads)
{
    return orc_attention_window(n_q, H_q, H_kv, d, q, qpos, L, K, V, out, nthreads, 0);
}
