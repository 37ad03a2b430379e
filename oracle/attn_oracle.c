/*
 * Float64 CPU oracle for exact attention.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * call this code.  The CUDA library never links, includes or calls it, and
 * this file includes nothing from the CUDA library.
 *
 * What it computes is the plain definition of attention, not the tiled
 * method: the method reaches this same result up to rounding order
 * ("FlashAttention: The Matrix You Never Have to Write Down", section
 * "What attention computes, in one page", the Attention(Q,K,V) equation;
 * section "Check it", the float64 exact_attention reference, which builds
 * the scores, masks the future, applies softmax and multiplies by V).
 *
 * For one query row q at absolute position p, against keys K[0..nk) and
 * values V[0..nk):
 *   visible keys  j : j < nk, and j <= p when causal (upper-left alignment,
 *                     section "Build it", note on non-square causal alignment)
 *   s_j  = scale * sum_c q_c K[j][c]
 *   m    = max_j s_j                      (stable softmax, section "What stops
 *                                          us: softmax needs the whole row")
 *   l    = sum_j exp(s_j - m)
 *   o    = sum_j exp(s_j - m) V[j] / l
 *   lse  = m + ln(l)                      (natural log of the scaled scores,
 *                                          as torch.logsumexp in "Check it")
 * A row with no visible key gets o = 0 and lse = -inf: the pages' stated
 * policy for an empty key sequence (section "Check it", the empty-key case).
 *
 * Every step is in double precision.  One row of scores (nk doubles) is held
 * per thread; the full query-by-key matrix is never built, because the long
 * workloads would need gigabytes per head for it.  Rows are independent and
 * are spread over OpenMP threads; each row's arithmetic is sequential in key
 * order, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Returns 0 on success, -1 on a bad argument, -2 if a row buffer could not be
 * allocated. */
int oracle_attention_rows(int64_t nk, int64_t d, int64_t dv,
                          const double *k, const double *v,
                          int64_t nrows, const double *q_rows,
                          const int64_t *q_pos, int causal, double scale,
                          double *o_rows, double *lse_rows)
{
    if (nk < 0 || d <= 0 || dv <= 0 || nrows < 0)
        return -1;
    if (nrows == 0)
        return 0;
    if (!q_rows || !o_rows || !lse_rows || (causal && !q_pos))
        return -1;
    if (nk > 0 && (!k || !v))
        return -1;

    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s)
                continue;
            const double *q = q_rows + r * d;
            double *o = o_rows + r * dv;

            /* how many keys this row may see */
            int64_t nvis = nk;
            if (causal) {
                int64_t p = q_pos[r];
                nvis = p < 0 ? 0 : (p + 1 < nk ? p + 1 : nk);
            }

            for (int64_t c = 0; c < dv; ++c)
                o[c] = 0.0;
            if (nvis == 0) {
                lse_rows[r] = -INFINITY;
                continue;
            }

            /* scores of this row */
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

            /* softmax weights against the row maximum, and the V blend */
            double l = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                double w = exp(s[j] - m);
                l += w;
                const double *vj = v + j * dv;
                for (int64_t c = 0; c < dv; ++c)
                    o[c] += w * vj[c];
            }
            for (int64_t c = 0; c < dv; ++c)
                o[c] /= l;
            lse_rows[r] = m + log(l);
        }
        free(s);
    }
    return failed ? -2 : 0;
}

/* Whole heads: q [bh, nq, d], k [bh, nk, d], v [bh, nk, dv] -> o [bh, nq, dv],
 * lse [bh, nq].  Query i sits at absolute position i. */
int oracle_attention(int64_t bh, int64_t nq, int64_t nk, int64_t d, int64_t dv,
                     const double *q, const double *k, const double *v,
                     int causal, double scale, double *o, double *lse)
{
    if (bh < 0 || nq < 0)
        return -1;
    if (bh == 0 || nq == 0)
        return 0;
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)nq);
    if (!pos)
        return -2;
    for (int64_t i = 0; i < nq; ++i)
        pos[i] = i;
    int rc = 0;
    for (int64_t h = 0; h < bh && rc == 0; ++h)
        rc = oracle_attention_rows(nk, d, dv, k ? k + h * nk * d : 0,
                                   v ? v + h * nk * dv : 0, nq, q + h * nq * d,
                                   pos, causal, scale, o + h * nq * dv,
                                   lse + h * nq);
    free(pos);
    return rc;
}

/* Number of threads the rows above run on (for reporting). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
