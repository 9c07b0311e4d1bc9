/*
 * attn_bwd_oracle.c -- CPU oracle for the gradients of the exact attention
 * forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; it gives the tests and the benchmark's CPU baseline an
 * independent, obviously correct answer for the backward pass.  It shares
 * no code, header, table or constant with the CUDA library.
 *
 * The pages name the backward pass without writing it out ("FlashAttention
 * v4 Blackwell pipeline 原理详解", pseudo-code panel, "backward idea", and
 * the CTA-role panel on the 2-CTA backward: two CTAs share a larger MMA
 * tile so that fewer dQ atomic additions are needed).  The plainest
 * reading is the vector-Jacobian product of the forward's definition: for
 * an upstream gradient dO of the output O, the gradients of
 * L = sum_{i,c} dO_ic O_ic with respect to Q, K and V.  Written out with
 * the chain rule, in fp64, for each (b, h) and each query row i:
 *
 *   s_ij  = scale * sum_c q_ic k_jc                  j in A(i)
 *   p_ij  = exp(s_ij - m_i) / l_i                    (three-pass softmax)
 *   dp_ij = sum_c dO_ic v_jc                         dL/dp_ij
 *   r_i   = sum_{j in A(i)} p_ij dp_ij
 *   ds_ij = p_ij (dp_ij - r_i)                       softmax Jacobian
 *   dV_j += p_ij dO_i
 *   dQ_i  = scale * sum_j ds_ij k_j
 *   dK_j += scale * ds_ij q_i
 *
 * with A(i) = {0..N-1}, or {0..i} when causal, as in the forward oracle.
 * r_i is formed from its definition (sum of p dp), not from O.
 *
 * Layout: q, k, v, dout, dq, dk, dv are [B, H, N, d] row-major fp64.
 * Return codes: 0 ok, -1 bad argument, -2 out of memory, -3 thread error.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *dout;
    int64_t N, d;
    int causal;
    double scale;
    int64_t head_begin, head_end; /* heads (b*H + h) of this thread */
    double *dq, *dk, *dv;
    int status;
} bwd_job;

/* All gradients of one head. */
static int one_head(const bwd_job *jb, int64_t bh, double *s, double *p, double *dp)
{
    const int64_t N = jb->N, d = jb->d;
    const double *Q = jb->q + bh * N * d, *K = jb->k + bh * N * d, *V = jb->v + bh * N * d;
    const double *dO = jb->dout + bh * N * d;
    double *dQ = jb->dq + bh * N * d, *dK = jb->dk + bh * N * d, *dV = jb->dv + bh * N * d;
    memset(dK, 0, sizeof(double) * (size_t)(N * d));
    memset(dV, 0, sizeof(double) * (size_t)(N * d));
    for (int64_t i = 0; i < N; ++i) {
        const double *qi = Q + i * d, *doi = dO + i * d;
        const int64_t nvis = jb->causal ? i + 1 : N;
        /* the forward's probabilities of row i, three passes */
        double m = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += qi[c] * K[j * d + c];
            s[j] = jb->scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            l += exp(s[j] - m);
        for (int64_t j = 0; j < nvis; ++j)
            p[j] = exp(s[j] - m) / l;
        /* dL/dp and the row's weighted sum r */
        double r = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += doi[c] * V[j * d + c];
            dp[j] = dot;
            r += p[j] * dp[j];
        }
        /* dV, and dS through the softmax Jacobian into dQ and dK */
        double *dqi = dQ + i * d;
        for (int64_t c = 0; c < d; ++c)
            dqi[c] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            const double ds = p[j] * (dp[j] - r);
            for (int64_t c = 0; c < d; ++c) {
                dV[j * d + c] += p[j] * doi[c];
                dqi[c] += jb->scale * ds * K[j * d + c];
                dK[j * d + c] += jb->scale * ds * qi[c];
            }
        }
    }
    return 0;
}

static void *run_bwd_job(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    const size_t n = (size_t)jb->N;
    double *buf = (double *)malloc(sizeof(double) * 3 * n);
    if (!buf) {
        jb->status = -2;
        return NULL;
    }
    for (int64_t bh = jb->head_begin; bh < jb->head_end; ++bh)
        one_head(jb, bh, buf, buf + n, buf + 2 * n);
    free(buf);
    jb->status = 0;
    return NULL;
}

/*
 * Gradients dq, dk, dv [B, H, N, d] of sum(dout * O) for the attention
 * forward on q, k, v.  Heads are split over nthreads POSIX threads; each
 * head is computed by one thread in a fixed order, so the result does not
 * depend on the thread count.
 */
int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
                    double *dq, double *dk, double *dv, int nthreads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || B <= 0 || H <= 0 || N <= 0 || d <= 0)
        return -1;
    const int64_t heads = B * H;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > heads)
        nthreads = (int)heads;
    bwd_job *jobs = (bwd_job *)calloc((size_t)nthreads, sizeof(bwd_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    int rc = 0, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        bwd_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->dout = dout;
        jb->N = N; jb->d = d;
        jb->causal = causal; jb->scale = scale;
        jb->head_begin = heads * t / nthreads;
        jb->head_end = heads * (t + 1) / nthreads;
        jb->dq = dq; jb->dk = dk; jb->dv = dv;
        jb->status = -3;
        if (t == 0)
            continue; /* the calling thread takes range 0 */
        if (pthread_create(&tids[t], NULL, run_bwd_job, jb) != 0) {
            rc = -3;
            break;
        }
        started = t;
    }
    if (rc == 0)
        run_bwd_job(&jobs[0]);
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
 * dQ only, for a list of query rows (flat ids (b*H + h)*N + i): each row's
 * gradient needs only that row's probabilities, so large shapes can be
 * checked on samples.  The same chain rule as oracle_attn_bwd, row by row:
 * p_ij from the three-pass softmax, dp_ij = dO_i . v_j, r_i = sum_j p_ij dp_ij,
 * dq_i = scale * sum_j p_ij (dp_ij - r_i) k_j.  dq is [nrows, d].
 * Rows are split over nthreads POSIX threads.
 */
typedef struct {
    const double *q, *k, *v, *dout;
    int64_t N, d;
    int causal;
    double scale;
    const int64_t *rows;
    int64_t begin, end;
    double *dq;
    int status;
} dq_job;

static void *run_dq_job(void *arg)
{
    dq_job *jb = (dq_job *)arg;
    const int64_t N = jb->N, d = jb->d;
    double *s = (double *)malloc(sizeof(double) * 2 * (size_t)N);
    if (!s) {
        jb->status = -2;
        return NULL;
    }
    double *dp = s + N;
    for (int64_t r = jb->begin; r < jb->end; ++r) {
        const int64_t flat = jb->rows[r], bh = flat / N, i = flat % N;
        const double *qi = jb->q + flat * d, *doi = jb->dout + flat * d;
        const double *K = jb->k + bh * N * d, *V = jb->v + bh * N * d;
        const int64_t nvis = jb->causal ? i + 1 : N;
        double m = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += qi[c] * K[j * d + c];
            s[j] = jb->scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nvis; ++j)
            l += exp(s[j] - m);
        double rr = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += doi[c] * V[j * d + c];
            dp[j] = dot;
            rr += exp(s[j] - m) / l * dot;
        }
        double *out = jb->dq + r * d;
        for (int64_t c = 0; c < d; ++c)
            out[c] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            const double ds = exp(s[j] - m) / l * (dp[j] - rr);
            for (int64_t c = 0; c < d; ++c)
                out[c] += jb->scale * ds * K[j * d + c];
        }
    }
    free(s);
    jb->status = 0;
    return NULL;
}

int oracle_attn_bwd_dq_rows(const double *q, const double *k, const double *v,
                            const double *dout, int64_t B, int64_t H, int64_t N, int64_t d,
                            int causal, double scale, const int64_t *rows, int64_t nrows,
                            double *dq, int nthreads)
{
    if (!q || !k || !v || !dout || !rows || !dq || B <= 0 || H <= 0 || N <= 0 || d <= 0 ||
        nrows < 0)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N)
            return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = nrows > 0 ? (int)nrows : 1;
    dq_job *jobs = (dq_job *)calloc((size_t)nthreads, sizeof(dq_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    int rc = 0, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        dq_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->dout = dout;
        jb->N = N; jb->d = d;
        jb->causal = causal; jb->scale = scale;
        jb->rows = rows;
        jb->begin = nrows * t / nthreads;
        jb->end = nrows * (t + 1) / nthreads;
        jb->dq = dq;
        jb->status = -3;
        if (t == 0)
            continue;
        if (pthread_create(&tids[t], NULL, run_dq_job, jb) != 0) {
            rc = -3;
            break;
        }
        started = t;
    }
    if (rc == 0)
        run_dq_job(&jobs[0]);
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
