/*
 * Float64 CPU oracle for exact attention with dropout on the attention
 * weights.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU legs call
 * this code.  The CUDA library never links, includes or calls it, and this
 * file includes nothing from the CUDA library.
 *
 * What the pages fix: the full algorithm, with dropout enabled, keeps the
 * pseudorandom generator's state so that the backward pass regenerates the
 * same dropout mask instead of storing a square mask ("Why FlashAttention
 * Can Avoid a Square Attention Array Without Making Attention Linear",
 * section "Backward can recreate tiles instead of retaining the square";
 * the first page's note on PyTorch's attention says dropout_p is applied as
 * given).  They fix neither the generator nor how its bits become a mask;
 * the readings taken here:
 *
 *   generator  Philox4x32 with 10 rounds, a counter-based generator (Salmon,
 *              Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *              1, 2, 3", SC 2011): a 128-bit counter and a 64-bit key give
 *              four 32-bit words, each round multiplying two counter words
 *              by fixed odd constants and mixing high and low halves with
 *              the other words and the key, the key bumped by two Weyl
 *              constants between rounds.
 *   blocks     one call covers a 4 x 4 block of the attention matrix of one
 *              (batch, head): counter = (key index / 4, query index / 4,
 *              batch*head index, offset), key = the 64-bit seed (low word
 *              first).  Element (i, j) takes byte j % 4 of word i % 4.
 *   keep       the element is kept when that byte is below
 *              t = floor((1 - p) * 256 + 1/2), 1 <= t <= 256, so its keep
 *              probability is t / 256; kept weights are scaled by 256 / t,
 *              so the mask has mean exactly one.
 *
 * Queries against a key set of another length (a chunk after a cache,
 * padding, packed sequences): query row i sits at position i + q_off and,
 * with causal masking, sees keys j <= i + q_off (none when that is
 * negative: O = 0, LSE = -inf, the empty-key policy); the mask stays
 * indexed by the row i and the key index j, so the offset moves only the
 * causal boundary, never a keep decision (a reading; the pages fix no mask
 * layout).
 *
 * With Z[i][j] in {0, 1} the keep decision and s = 256 / t, the forward
 * output is, over the visible keys of row i (causal: j <= i + q_off),
 *
 *     O[i] = s * sum_j exp(x_ij - m_i) Z[i][j] V[j] / l_i,
 *     l_i  = sum_j exp(x_ij - m_i),   LSE[i] = m_i + ln l_i,
 *
 * x_ij = scale * q_i . k_j: the normalisation is that of the softmax without
 * dropout, and LSE is unchanged by it.  The gradient of
 * loss = sum dO * O, by the chain rule (P = exp(x - LSE)):
 *
 *     dV[j]    = s * sum_i P[i][j] Z[i][j] dO[i]
 *     dP[i][j] = s * Z[i][j] (dO[i] . V[j])
 *     D[i]     = sum_j P[i][j] dP[i][j]   ( = dO[i] . O[i] )
 *     dS[i][j] = P[i][j] (dP[i][j] - D[i])
 *     dQ[i]    = scale * sum_j dS[i][j] K[j],  dK[j] = scale * sum_i dS[i][j] Q[i].
 *
 * Every step is in double precision and sequential within a head; heads
 * are independent and are spread over OpenMP threads by the callers'
 * batching (one head per call here keeps the code plain).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* Philox4x32-10: out = the generator's four words for counter ctr, key key. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;   /* round multipliers */
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;   /* key bumps (Weyl) */
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const uint64_t p0 = (uint64_t)M0 * c0;
        const uint64_t p1 = (uint64_t)M1 * c2;
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* Keep decision Z[i][j] of (batch*head) bh for the given seed, offset and t. */
static int keep(int64_t bh, int64_t i, int64_t j, uint64_t seed, uint32_t offset, int t)
{
    const uint32_t ctr[4] = {(uint32_t)(j / 4), (uint32_t)(i / 4), (uint32_t)bh, offset};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    const uint32_t byte = (w[i % 4] >> (8 * (j % 4))) & 0xFFu;
    return byte < (uint32_t)t;
}

/* The keep mask of one head, mask[i * nk + j] in {0, 1} (small shapes). */
int oracle_dropout_mask(int64_t bh, int64_t nq, int64_t nk, uint64_t seed, uint32_t offset,
                        int t, uint8_t *mask)
{
    if (nq < 0 || nk < 0 || t < 1 || t > 256 || (nq * nk > 0 && !mask))
        return -1;
    for (int64_t i = 0; i < nq; ++i)
        for (int64_t j = 0; j < nk; ++j)
            mask[i * nk + j] = (uint8_t)keep(bh, i, j, seed, offset, t);
    return 0;
}

static int64_t visible(int64_t i, int64_t nk, int causal, int64_t q_off)
{
    if (!causal)
        return nk;
    const int64_t last = i + 1 + q_off;   /* keys 0 .. i + q_off */
    return last <= 0 ? 0 : (last < nk ? last : nk);
}

/* Forward with dropout for one head (query i at position i + q_off). */
int oracle_attention_dropout(int64_t bh, int64_t nq, int64_t nk, int64_t d, int64_t dv,
                             const double *q, const double *k, const double *v, int causal,
                             int64_t q_off, double scale, uint64_t seed, uint32_t offset, int t,
                             double *o, double *lse)
{
    if (nq < 0 || nk < 0 || d <= 0 || dv <= 0 || t < 1 || t > 256)
        return -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    if (!x)
        return -2;
    const double s = 256.0 / (double)t;
    for (int64_t i = 0; i < nq; ++i) {
        double *oi = o + i * dv;
        for (int64_t c = 0; c < dv; ++c)
            oi[c] = 0.0;
        const int64_t nvis = visible(i, nk, causal, q_off);
        if (nvis == 0) {
            lse[i] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += q[i * d + c] * k[j * d + c];
            x[j] = scale * dot;
            if (x[j] > m)
                m = x[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            const double e = exp(x[j] - m);
            l += e;
            if (keep(bh, i, j, seed, offset, t))
                for (int64_t c = 0; c < dv; ++c)
                    oi[c] += e * v[j * dv + c];
        }
        for (int64_t c = 0; c < dv; ++c)
            oi[c] *= s / l;
        lse[i] = m + log(l);
    }
    free(x);
    return 0;
}

/* Gradients with dropout for one head: dq [nq, d], dk [nk, d], dvv [nk, dv]
 * (written, not accumulated into). */
int oracle_attention_dropout_grad(int64_t bh, int64_t nq, int64_t nk, int64_t d, int64_t dv,
                                  const double *q, const double *k, const double *v,
                                  const double *dout, int causal, int64_t q_off, double scale,
                                  uint64_t seed, uint32_t offset, int t, double *dq, double *dk,
                                  double *dvv)
{
    if (nq < 0 || nk < 0 || d <= 0 || dv <= 0 || t < 1 || t > 256)
        return -1;
    double *o = (double *)malloc(sizeof(double) * (size_t)(nq > 0 ? nq * dv : 1));
    double *lse = (double *)malloc(sizeof(double) * (size_t)(nq > 0 ? nq : 1));
    double *pr = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    int rc = 0;
    if (!o || !lse || !pr || !dp) {
        rc = -2;
        goto done;
    }
    rc = oracle_attention_dropout(bh, nq, nk, d, dv, q, k, v, causal, q_off, scale, seed, offset,
                                  t, o, lse);
    if (rc != 0)
        goto done;
    const double s = 256.0 / (double)t;
    for (int64_t x = 0; x < nq * d; ++x)
        dq[x] = 0.0;
    for (int64_t x = 0; x < nk * d; ++x)
        dk[x] = 0.0;
    for (int64_t x = 0; x < nk * dv; ++x)
        dvv[x] = 0.0;
    for (int64_t i = 0; i < nq; ++i) {
        const int64_t nvis = visible(i, nk, causal, q_off);
        if (nvis == 0)
            continue;
        const double *gi = dout + i * dv;
        double dd = 0.0;   /* D[i] = dO[i] . O[i] */
        for (int64_t c = 0; c < dv; ++c)
            dd += gi[c] * o[i * dv + c];
        for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += q[i * d + c] * k[j * d + c];
            pr[j] = exp(scale * dot - lse[i]);
            const int z = keep(bh, i, j, seed, offset, t);
            double gv = 0.0;
            for (int64_t c = 0; c < dv; ++c)
                gv += gi[c] * v[j * dv + c];
            dp[j] = z ? s * gv : 0.0;
            if (z)
                for (int64_t c = 0; c < dv; ++c)
                    dvv[j * dv + c] += s * pr[j] * gi[c];
        }
        for (int64_t j = 0; j < nvis; ++j) {
            const double ds = pr[j] * (dp[j] - dd);
            for (int64_t c = 0; c < d; ++c) {
                dq[i * d + c] += scale * ds * k[j * d + c];
                dk[j * d + c] += scale * ds * q[i * d + c];
            }
        }
    }
done:
    free(o);
    free(lse);
    free(pr);
    free(dp);
    return rc;
}
