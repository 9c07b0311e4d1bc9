/*
 * attn_oracle.c -- CPU oracle for the exact attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; it exists so the tests, the smoke check and the CPU
 * baseline of the benchmark have an independent, obviously correct answer
 * to compare the GPU kernels against.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes is the plain definition of attention, in fp64, with the
 * three-pass "safe" softmax:
 *
 *   s_ij  = scale * sum_c q_ic k_jc          for j in A(i)
 *   m_i   = max_{j in A(i)} s_ij                               (pass 1)
 *   l_i   = sum_{j in A(i)} exp(s_ij - m_i)                    (pass 2)
 *   p_ij  = exp(s_ij - m_i) / l_i,  p_ij = 0 for j not in A(i) (pass 3)
 *   o_ic  = sum_j p_ij v_jc
 *   lse_i = m_i + ln(l_i)
 *
 * A(i) = {0..N-1}, or {0..i} when the causal mask is on (key j visible to
 * query i iff j <= i).
 *
 * Sources:
 *  - "flash attention v2 论文" search page, the FlashAttention abstract
 *    snippet: the method is not an approximation; its output equals that of
 *    conventional attention.  So the exact result is the definition above.
 *  - same page, the "(Safe) Softmax: 3-pass" outline: max pass, sum pass,
 *    divide pass -- the order the loops below follow.
 *  - "FlashAttention v4 Blackwell pipeline 原理详解", pseudo-code panel:
 *    "final normalize O = acc / l" -- l is the softmax denominator.
 *  - The pages never define the logsumexp; it is read here as the natural
 *    log of the denominator of the *scaled* logits (lse = m + ln l).
 *
 * Layout: q, k, v are [B, H, N, d] row-major fp64; element (b,h,n,c) sits at
 * ((b*H + h)*N + n)*d + c.  Outputs o [rows, d] and lse [rows] in the order
 * rows are requested.
 *
 * Return codes: 0 ok, -1 bad argument, -2 out of memory, -3 thread error.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v;
    int64_t H, N, d;
    int causal;
    double scale;
    const int64_t *rows; /* flat row ids: (b*H + h)*N + i */
    int64_t row_begin, row_end;
    double *o, *lse;
    int status;
} oracle_job;

/* One query row, the three passes written out in full. */
static void one_row(const oracle_job *jb, int64_t flat, double *s, double *o_out,
                    double *lse_out)
{
    const int64_t N = jb->N, d = jb->d;
    const int64_t bh = flat / N;
    const int64_t i = flat % N;
    const double *qi = jb->q + flat * d;
    const double *K = jb->k + bh * N * d;
    const double *V = jb->v + bh * N * d;
    const int64_t nvis = jb->causal ? i + 1 : N; /* |A(i)|: keys 0..nvis-1 */

    /* logits and pass 1: the row maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += qi[c] * K[j * d + c];
        s[j] = jb->scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    /* pass 2: the denominator */
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j)
        l += exp(s[j] - m);
    /* pass 3: probabilities and the weighted sum of values */
    for (int64_t c = 0; c < d; ++c)
        o_out[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        const double p = exp(s[j] - m) / l;
        for (int64_t c = 0; c < d; ++c)
            o_out[c] += p * V[j * d + c];
    }
    *lse_out = m + log(l);
}

static void *run_job(void *arg)
{
    oracle_job *jb = (oracle_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)jb->N);
    if (!s) {
        jb->status = -2;
        return NULL;
    }
    for (int64_t r = jb->row_begin; r < jb->row_end; ++r) {
        const int64_t flat = jb->rows ? jb->rows[r] : r;
        one_row(jb, flat, s, jb->o + r * jb->d, jb->lse + r);
    }
    free(s);
    jb->status = 0;
    return NULL;
}

/*
 * Attention forward for a list of rows (or all B*H*N rows when rows == NULL,
 * in which case nrows must equal B*H*N).  Work is split over nthreads
 * POSIX threads by contiguous ranges of the row list; each row is computed
 * independently, so the result does not depend on the thread count.
 */
int oracle_attn_fwd_rows(const double *q, const double *k, const double *v, int64_t B,
                         int64_t H, int64_t N, int64_t d, int causal, double scale,
                         const int64_t *rows, int64_t nrows, double *o, double *lse,
                         int nthreads)
{
    if (!q || !k || !v || !o || !lse || B <= 0 || H <= 0 || N <= 0 || d <= 0 || nrows < 0)
        return -1;
    const int64_t total = B * H * N;
    if (!rows && nrows != total)
        return -1;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= total)
                return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = nrows > 0 ? (int)nrows : 1;

    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    int rc = 0, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v;
        jb->H = H; jb->N = N; jb->d = d;
        jb->causal = causal; jb->scale = scale;
        jb->rows = rows;
        jb->row_begin = nrows * t / nthreads;
        jb->row_end = nrows * (t + 1) / nthreads;
        jb->o = o; jb->lse = lse;
        jb->status = -3;
        if (t == 0)
            continue; /* the calling thread takes range 0 */
        if (pthread_create(&tids[t], NULL, run_job, jb) != 0) {
            rc = -3;
            break;
        }
        started = t;
    }
    if (rc == 0)
        run_job(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tids[t], NULL);
    if (rc == 0)
        for (int t = 0; t < nthreads; ++t)
            if (jobs[t].status != 0)
                rc = jobs[t].status;
    free(jobs);
    free(tids);
    return rc;
}

/*
 * The full probability matrix P [B, H, N, N] (masked entries exactly 0),
 * for small shapes only: it lets the tests check the softmax itself (rows
 * sum to one, masked entries are zero) and not just its product with V.
 */
int oracle_attn_probs(const double *q, const double *k, int64_t B, int64_t H, int64_t N,
                      int64_t d, int causal, double scale, double *p)
{
    if (!q || !k || !p || B <= 0 || H <= 0 || N <= 0 || d <= 0)
        return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    if (!s)
        return -2;
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const double *K = k + bh * N * d;
        for (int64_t i = 0; i < N; ++i) {
            const double *qi = q + (bh * N + i) * d;
            double *prow = p + (bh * N + i) * N;
            const int64_t nvis = causal ? i + 1 : N;
            double m = -INFINITY;
            for (int64_t j = 0; j < nvis; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += qi[c] * K[j * d + c];
                s[j] = scale * dot;
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nvis; ++j)
                l += exp(s[j] - m);
            for (int64_t j = 0; j < N; ++j)
                prow[j] = (j < nvis) ? exp(s[j] - m) / l : 0.0;
        }
    }
    free(s);
    return 0;
}
