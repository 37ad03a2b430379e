"""Pins of the float64 dropout oracle, each a function of the compiled
oracle library so the mutant tests can run them against planted mistakes.

What they pin it to, from outside its own code: the generator's published
known-answer vectors; the exact reduction to the dropout-free oracle at
p = 0 (also with queries at shifted positions, against the plain oracle's
rows at those positions); the binomial law of the keep rate; the
unbiasedness the 256 / t scale exists for; finite differences of the loss
with the mask held fixed (also with shifted queries).
"""
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "philox4x32_10_kat.txt")


def kat_rows():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(x, 16) for x in line.split()]
        rows.append((w[:4], w[4:6], w[6:10]))
    return rows


def rand_head(tq, tk, d, dv, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((tq, d)), r.standard_normal((tk, d)), r.standard_normal((tk, dv)),
            r.standard_normal((tq, dv)))


def pin_philox_known_answers(lib):
    rows = kat_rows()
    assert len(rows) == 3
    for ctr, key, want in rows:
        assert [int(x) for x in oracle.philox4x32_10(ctr, key, lib=lib)] == want


def pin_no_dropout_is_plain_attention(lib):
    """p = 0 keeps every weight with scale 1: the plain oracle's O, LSE and
    gradients (the plain oracle from the same library build)."""
    q, k, v, g = rand_head(37, 37, 8, 6, 1)
    for causal in (False, True):
        o, lse = oracle.attention_dropout(q, k, v, 5, 99, 3, 0.0, causal=causal, lib=lib)
        o2, lse2 = oracle.attention(q, k, v, causal=causal, lib=lib)
        assert np.abs(o - o2).max() < 1e-12 and np.abs(lse - lse2).max() < 1e-12
        gq, gk, gv = oracle.attention_dropout_grad(q, k, v, g, 5, 99, 3, 0.0, causal=causal, lib=lib)
        hq, hk, hv = oracle.attention_grad(q, k, v, g, causal=causal, lib=lib)
        for a, b in ((gq, hq), (gk, hk), (gv, hv)):
            assert np.abs(a - b).max() < 1e-11


def pin_keep_rate_is_binomial(lib):
    """Over 512 x 512 elements the kept fraction is t / 256 within 5 sigma
    for several p, heads, seeds and offsets; neighbours are uncorrelated;
    another offset draws another mask, the same one the same."""
    n = 512 * 512
    seen = []
    for p, bh, seed, off in [(0.1, 0, 1, 0), (0.5, 7, 2, 0), (0.5, 7, 2, 1), (0.9, 3, 2 ** 40, 9)]:
        m = oracle.dropout_mask(bh, 512, 512, seed, off, p, lib=lib)
        frac = oracle.dropout_threshold(p) / 256.0
        sigma = np.sqrt(frac * (1 - frac) / n)
        assert abs(m.mean() - frac) < 5 * sigma, (p, m.mean(), frac)
        a = m.astype(np.float64) - m.mean()
        for nb in (a[:, 1:] * a[:, :-1], a[1:, :] * a[:-1, :]):
            assert abs(nb.mean()) < 6 * frac * (1 - frac) / np.sqrt(nb.size)
        seen.append(m)
    assert not np.array_equal(seen[1], seen[2])
    assert np.array_equal(seen[1], oracle.dropout_mask(7, 512, 512, 2, 0, 0.5, lib=lib))


def pin_dropout_is_unbiased(lib):
    """Averaged over many masks (offsets) the output is the dropout-free
    output (E[Z] 256 / t = 1), element by element within 5 standard errors
    of the sample's own spread."""
    q, k, v, _ = rand_head(8, 24, 8, 5, 2)
    for causal in (False, True):
        o0, _ = oracle.attention(q, k, v, causal=causal, lib=lib)
        draws = np.stack([oracle.attention_dropout(q, k, v, 0, 77, off, 0.3, causal=causal,
                                                   lib=lib)[0] for off in range(1500)])
        mean, se = draws.mean(0), draws.std(0) / np.sqrt(len(draws))
        assert np.all(np.abs(mean - o0) <= 5 * se + 1e-12)


def pin_gradient_matches_finite_differences(lib):
    """With seed and offset fixed the mask is fixed and the loss sum(dO * O)
    is smooth: central differences of the forward give dQ, dK, dV."""
    q, k, v, g = rand_head(11, 13, 4, 3, 3)
    args = (2, 12345, 6, 0.4)
    h = 1e-6
    r = np.random.default_rng(4)
    for causal in (False, True):
        grads = oracle.attention_dropout_grad(q, k, v, g, *args, causal=causal, lib=lib)

        def loss(x3):
            return float(np.sum(g * oracle.attention_dropout(*x3, *args, causal=causal, lib=lib)[0]))

        for pos in range(3):
            x = (q, k, v)[pos]
            for _ in range(12):
                idx = tuple(int(r.integers(0, s)) for s in x.shape)
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                a = [q, k, v]
                a[pos] = xp
                lp = loss(a)
                a[pos] = xm
                lm = loss(a)
                fd = (lp - lm) / (2 * h)
                gx = grads[pos][idx]
                assert abs(fd - gx) <= 1e-6 * max(1.0, abs(fd)), ("qkv"[pos], idx, fd, gx)


def pin_offset_moves_only_the_causal_boundary(lib):
    """Queries at shifted positions (row i at i + q_offset): at p = 0 every
    row is the plain oracle's row at that position (rows before the first
    key empty: O = 0, LSE = -inf); without causal masking the offset changes
    nothing (the mask is indexed by row and key, not by position); an offset
    past the last key sees every key, as the unmasked call does with the
    same mask."""
    q, k, v, _ = rand_head(9, 20, 6, 5, 5)
    for off in (-4, 0, 3, 11):
        o, lse = oracle.attention_dropout(q, k, v, 3, 17, 2, 0.0, causal=True, lib=lib, q_offset=off)
        pos = np.arange(9) + off
        o2, l2 = oracle.attention_rows(q, pos, k, v, causal=True, lib=lib)
        seen = np.isfinite(l2)
        assert np.abs(o[seen] - o2[seen]).max() < 1e-12
        assert np.abs(lse[seen] - l2[seen]).max() < 1e-12
        assert np.all(o[~seen] == 0.0) and np.all(np.isneginf(lse[~seen]))
    base = oracle.attention_dropout(q, k, v, 3, 17, 2, 0.3, causal=False, lib=lib)
    for off in (-4, 5, 11):
        o, lse = oracle.attention_dropout(q, k, v, 3, 17, 2, 0.3, causal=False, lib=lib, q_offset=off)
        assert np.array_equal(o, base[0]) and np.array_equal(lse, base[1])
    o, lse = oracle.attention_dropout(q, k, v, 3, 17, 2, 0.3, causal=True, lib=lib, q_offset=20)
    assert np.abs(o - base[0]).max() < 1e-13 and np.abs(lse - base[1]).max() < 1e-13


def pin_gradient_with_offset_matches_finite_differences(lib):
    """Finite differences of sum(dO * O) with the queries shifted (some rows
    see nothing, others see all keys) and the mask fixed."""
    q, k, v, g = rand_head(7, 10, 4, 3, 6)
    h = 1e-6
    r = np.random.default_rng(7)
    for off in (-3, 4):
        args = (1, 999, 4, 0.35)
        grads = oracle.attention_dropout_grad(q, k, v, g, *args, causal=True, lib=lib, q_offset=off)

        def loss(x3):
            return float(np.sum(g * oracle.attention_dropout(*x3, *args, causal=True, lib=lib,
                                                             q_offset=off)[0]))

        for pos in range(3):
            x = (q, k, v)[pos]
            for _ in range(10):
                idx = tuple(int(r.integers(0, s)) for s in x.shape)
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                a = [q, k, v]
                a[pos] = xp
                lp = loss(a)
                a[pos] = xm
                lm = loss(a)
                fd = (lp - lm) / (2 * h)
                assert abs(fd - grads[pos][idx]) <= 1e-6 * max(1.0, abs(fd)), ("qkv"[pos], off, idx)


ALL_DROPOUT_PINS = [pin_philox_known_answers, pin_no_dropout_is_plain_attention,
                    pin_keep_rate_is_binomial, pin_dropout_is_unbiased,
                    pin_gradient_matches_finite_differences,
                    pin_offset_moves_only_the_causal_boundary,
                    pin_gradient_with_offset_matches_finite_differences]
