"""Pins of the float64 dropout oracle (CPU only).

The pages say only that, with dropout, the generator's state is kept so the
backward pass regenerates the same mask ("Why FlashAttention Can Avoid a
Square Attention Array Without Making Attention Linear", section "Backward
can recreate tiles instead of retaining the square").  The oracle's
generator, keep rule and gradients are pinned here against things outside
its own code: the generator's published known-answer vectors, the exact
reduction to the dropout-free oracle at p = 0, the keep rate's binomial
law, the unbiasedness the 256 / t scale is there for, and finite
differences of the loss with the mask held fixed.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def kat_rows():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(x, 16) for x in line.split()]
        rows.append((w[:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answers():
    rows = kat_rows()
    assert len(rows) == 3
    for ctr, key, want in rows:
        assert [int(x) for x in oracle.philox4x32_10(ctr, key)] == want


def rand_head(tq, tk, d, dv, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((tq, d)), r.standard_normal((tk, d)), r.standard_normal((tk, dv)),
            r.standard_normal((tq, dv)))


@pytest.mark.parametrize("causal", [False, True])
def test_no_dropout_is_plain_attention(causal):
    """p = 0 keeps every weight with scale 1: the plain oracle's O, LSE and
    gradients."""
    q, k, v, g = rand_head(37, 37, 8, 6, 1)
    o, lse = oracle.attention_dropout(q, k, v, 5, 99, 3, 0.0, causal=causal)
    o2, lse2 = oracle.attention(q, k, v, causal=causal)
    assert np.abs(o - o2).max() < 1e-12 and np.abs(lse - lse2).max() < 1e-12
    gq, gk, gv = oracle.attention_dropout_grad(q, k, v, g, 5, 99, 3, 0.0, causal=causal)
    hq, hk, hv = oracle.attention_grad(q, k, v, g, causal=causal)
    for a, b in ((gq, hq), (gk, hk), (gv, hv)):
        assert np.abs(a - b).max() < 1e-11


def test_keep_rate_is_binomial():
    """Over 512 x 512 elements the kept fraction is t / 256 within 5 sigma,
    for several p, heads, seeds and offsets; masks differ between them."""
    n = 512 * 512
    seen = []
    for p, bh, seed, off in [(0.1, 0, 1, 0), (0.5, 7, 2, 0), (0.5, 7, 2, 1), (0.9, 3, 2 ** 40, 9)]:
        m = oracle.dropout_mask(bh, 512, 512, seed, off, p)
        frac = oracle.dropout_threshold(p) / 256.0
        sigma = np.sqrt(frac * (1 - frac) / n)
        assert abs(m.mean() - frac) < 5 * sigma, (p, m.mean(), frac)
        # neighbours (same row, next column; same column, next row) are uncorrelated
        a = m.astype(np.float64) - m.mean()
        for nb in (a[:, 1:] * a[:, :-1], a[1:, :] * a[:-1, :]):
            assert abs(nb.mean()) < 6 * frac * (1 - frac) / np.sqrt(nb.size)
        seen.append(m)
    assert not np.array_equal(seen[1], seen[2])        # another offset, another mask
    assert np.array_equal(seen[1], oracle.dropout_mask(7, 512, 512, 2, 0, 0.5))   # regenerated


def test_threshold_reading():
    """t = floor((1 - p) * 256 + 1/2): halves round up (not to even)."""
    assert oracle.dropout_threshold(1 - 128.5 / 256) == 129
    assert oracle.dropout_threshold(0.0) == 256
    assert oracle.dropout_threshold(0.1) == 230
    assert oracle.dropout_threshold(0.5) == 128
    for bad in (1.0, -0.1, 0.999):
        with pytest.raises(ValueError):
            oracle.dropout_threshold(bad)


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_is_unbiased(causal):
    """Averaged over many masks (offsets) the output is the dropout-free
    output: E[Z] s = 1.  Checked element by element against the sample's
    own standard error."""
    q, k, v, _ = rand_head(8, 24, 8, 5, 2)
    o0, _ = oracle.attention(q, k, v, causal=causal)
    draws = np.stack([oracle.attention_dropout(q, k, v, 0, 77, off, 0.3, causal=causal)[0]
                      for off in range(1500)])
    mean, se = draws.mean(0), draws.std(0) / np.sqrt(len(draws))
    assert np.all(np.abs(mean - o0) <= 5 * se + 1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_gradient_matches_finite_differences(causal):
    """With the seed and offset fixed the mask is fixed and the loss
    sum(dO * O) is smooth: central differences of the forward oracle give
    the gradient oracle's dQ, dK, dV."""
    q, k, v, g = rand_head(11, 13, 4, 3, 3)
    args = (2, 12345, 6, 0.4)
    gq, gk, gv = oracle.attention_dropout_grad(q, k, v, g, *args, causal=causal)

    def loss(q_, k_, v_):
        return float(np.sum(g * oracle.attention_dropout(q_, k_, v_, *args, causal=causal)[0]))

    h = 1e-6
    r = np.random.default_rng(4)
    for name, x, gx in (("q", q, gq), ("k", k, gk), ("v", v, gv)):
        for _ in range(12):
            idx = tuple(int(r.integers(0, s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            parts = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}
            a = list(parts[name])
            pos = "qkv".index(name)
            a[pos] = xp
            lp = loss(*a)
            a[pos] = xm
            lm = loss(*a)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - gx[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, gx[idx])
