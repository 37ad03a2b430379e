/*
 * Float64 CPU oracle for the gradients of exact attention.
 * TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU legs call
 * this code.  The CUDA library never links, includes or calls it, and this
 * file includes nothing from the CUDA library.
 *
 * The pages say what a backward pass must do — keep Q, K, V, the output O
 * and the per-row statistics L, and rebuild the score and probability tiles
 * from them instead of storing the square ("FlashAttention: The Matrix You
 * Never Have to Write Down", section "The forward pass is only half of it";
 * "Why FlashAttention Can Avoid a Square Attention Array Without Making
 * Attention Linear", section "Backward can recreate tiles instead of
 * retaining the square") — but print no gradient formulas.  What is
 * computed here is the plain definition: the gradient of the scalar
 *
 *     loss = sum_{i,c} dO[i][c] * O[i][c],   O = softmax(scale * Q K^T) V
 *
 * (rows masked as in the forward oracle: key j visible to query i iff
 * j < nk and, when causal, j <= i) with respect to Q, K and V.  By the chain
 * rule, with P the row-normalised softmax weights over the visible keys:
 *
 *     dV[j]    = sum_i P[i][j] dO[i]
 *     dP[i][j] = dO[i] . V[j]
 *     D[i]     = sum_j P[i][j] dP[i][j]  ( = dO[i] . O[i] )
 *     dS[i][j] = P[i][j] (dP[i][j] - D[i])      (softmax Jacobian)
 *     dQ[i]    = scale * sum_j dS[i][j] K[j]
 *     dK[j]    = scale * sum_i dS[i][j] Q[i]
 *
 * Masked (invisible) pairs have P = 0 and contribute nothing.  P[i][j] is
 * taken as exp(s_ij - lse_i) with lse_i = m_i + ln l_i the row's
 * log-sum-exp, which is the same softmax written with the row statistics
 * the forward pass emits.
 *
 * Two passes, each embarrassingly parallel and without a query-by-key
 * matrix: rows of queries (dQ, lse, D), then rows of keys (dK, dV), the
 * second reading the per-query lse and D of the first.  Every step is in
 * double precision and sequential in key (or query) order within a row, so
 * the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int64_t visible_keys(int64_t pos, int64_t nk, int causal)
{
    if (!causal)
        return nk;
    if (pos < 0)
        return 0;
    return pos + 1 < nk ? pos + 1 : nk;
}

/*
 * Pass over query rows.  For each selected query row (position q_pos[r],
 * values q_rows[r], upstream gradient dout_rows[r]) against all keys of the
 * head: dq_rows[r], and the row's lse and D.  A row with no visible key gets
 * dq = 0, lse = -inf and D = 0.
 * Returns 0, -1 on a bad argument, -2 if a row buffer could not be allocated.
 */
int oracle_grad_query_rows(int64_t nk, int64_t d, int64_t dv,
                           const double *k, const double *v,
                           int64_t nrows, const double *q_rows, const double *dout_rows,
                           const int64_t *q_pos, int causal, double scale,
                           double *dq_rows, double *lse_rows, double *delta_rows)
{
    if (nk < 0 || d <= 0 || dv <= 0 || nrows < 0)
        return -1;
    if (nrows == 0)
        return 0;
    if (!q_rows || !dout_rows || !dq_rows || !lse_rows || !delta_rows || (causal && !q_pos))
        return -1;
    if (nk > 0 && (!k || !v))
        return -1;

    int failed = 0;
#pragma omp parallel
    {
        /* scores, then weights, of one row; and the row's output */
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        double *o = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!s || !o) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s || !o)
                continue;
            const double *q = q_rows + r * d;
            const double *g = dout_rows + r * dv;
            double *dq = dq_rows + r * d;
            for (int64_t c = 0; c < d; ++c)
                dq[c] = 0.0;
            const int64_t nvis = visible_keys(causal ? q_pos[r] : 0, nk, causal);
            if (nvis == 0) {
                lse_rows[r] = -INFINITY;
                delta_rows[r] = 0.0;
                continue;
            }
            /* forward quantities of the row: scores, max, sum, lse, O */
            double m = -INFINITY;
            for (int64_t j = 0; j < nvis; ++j) {
                const double *kj = k + j * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += q[c] * kj[c];
                s[j] = scale * dot;
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nvis; ++j)
                l += exp(s[j] - m);
            const double lse = m + log(l);
            for (int64_t c = 0; c < dv; ++c)
                o[c] = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                s[j] = exp(s[j] - lse);            /* P[i][j] */
                const double *vj = v + j * dv;
                for (int64_t c = 0; c < dv; ++c)
                    o[c] += s[j] * vj[c];
            }
            /* D = dO . O */
            double delta = 0.0;
            for (int64_t c = 0; c < dv; ++c)
                delta += g[c] * o[c];
            /* dQ = scale * sum_j P (dO . V_j - D) K_j */
            for (int64_t j = 0; j < nvis; ++j) {
                const double *vj = v + j * dv;
                double dp = 0.0;
                for (int64_t c = 0; c < dv; ++c)
                    dp += g[c] * vj[c];
                const double ds = s[j] * (dp - delta);
                const double *kj = k + j * d;
                for (int64_t c = 0; c < d; ++c)
                    dq[c] += scale * ds * kj[c];
            }
            lse_rows[r] = lse;
            delta_rows[r] = delta;
        }
        free(s);
        free(o);
    }
    return failed ? -2 : 0;
}

/*
 * Pass over key rows.  For each selected key row (position k_pos[r], values
 * k_rows[r] and v_rows[r]) against all nq queries of the head (q, dout, and
 * their lse and delta from oracle_grad_query_rows): dk_rows[r], dv_rows[r].
 * Query i sees key j when j < nk_total (the caller only passes real keys)
 * and, when causal, j <= i.  Queries with lse = -inf see nothing.
 */
int oracle_grad_key_rows(int64_t nq, int64_t d, int64_t dv,
                         const double *q, const double *dout,
                         const double *lse, const double *delta,
                         int64_t nrows, const double *k_rows, const double *v_rows,
                         const int64_t *k_pos, int causal, double scale,
                         double *dk_rows, double *dv_rows)
{
    if (nq < 0 || d <= 0 || dv <= 0 || nrows < 0)
        return -1;
    if (nrows == 0)
        return 0;
    if (!k_rows || !v_rows || !dk_rows || !dv_rows || (causal && !k_pos))
        return -1;
    if (nq > 0 && (!q || !dout || !lse || !delta))
        return -1;

#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < nrows; ++r) {
        const double *kj = k_rows + r * d;
        const double *vj = v_rows + r * dv;
        double *dk = dk_rows + r * d;
        double *dvr = dv_rows + r * dv;
        for (int64_t c = 0; c < d; ++c)
            dk[c] = 0.0;
        for (int64_t c = 0; c < dv; ++c)
            dvr[c] = 0.0;
        const int64_t first = causal ? (k_pos[r] < 0 ? 0 : k_pos[r]) : 0;
        for (int64_t i = first; i < nq; ++i) {
            if (lse[i] == -INFINITY)
                continue;
            const double *qi = q + i * d;
            const double *g = dout + i * dv;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += qi[c] * kj[c];
            const double p = exp(scale * dot - lse[i]);      /* P[i][j] */
            double dp = 0.0;
            for (int64_t c = 0; c < dv; ++c)
                dp += g[c] * vj[c];
            const double ds = p * (dp - delta[i]);
            for (int64_t c = 0; c < dv; ++c)
                dvr[c] += p * g[c];
            for (int64_t c = 0; c < d; ++c)
                dk[c] += scale * ds * qi[c];
        }
    }
    return 0;
}

/*
 * Whole heads: q [bh, nq, d], k [bh, nk, d], v [bh, nk, dv], dout [bh, nq, dv]
 * -> dq [bh, nq, d], dk [bh, nk, d], dvv [bh, nk, dv].  Query i sits at
 * position i and key j at position j.
 */
int oracle_attention_grad(int64_t bh, int64_t nq, int64_t nk, int64_t d, int64_t dv,
                          const double *q, const double *k, const double *v,
                          const double *dout, int causal, double scale,
                          double *dq, double *dk, double *dvv)
{
    if (bh < 0 || nq < 0 || nk < 0)
        return -1;
    if (bh == 0)
        return 0;
    const int64_t nmax = nq > nk ? nq : nk;
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nmax > 0 ? nmax : 1));
    double *lse = (double *)malloc(sizeof(double) * (size_t)(nq > 0 ? nq : 1));
    double *delta = (double *)malloc(sizeof(double) * (size_t)(nq > 0 ? nq : 1));
    if (!pos || !lse || !delta) {
        free(pos);
        free(lse);
        free(delta);
        return -2;
    }
    for (int64_t i = 0; i < nmax; ++i)
        pos[i] = i;
    int rc = 0;
    for (int64_t h = 0; h < bh && rc == 0; ++h) {
        rc = oracle_grad_query_rows(nk, d, dv, k + h * nk * d, v + h * nk * dv, nq,
                                    q + h * nq * d, dout + h * nq * dv, pos, causal, scale,
                                    dq + h * nq * d, lse, delta);
        if (rc == 0)
            rc = oracle_grad_key_rows(nq, d, dv, q + h * nq * d, dout + h * nq * dv, lse,
                                      delta, nk, k + h * nk * d, v + h * nk * dv, pos,
                                      causal, scale, dk + h * nk * d, dvv + h * nk * dv);
    }
    free(pos);
    free(lse);
    free(delta);
    return rc;
}
