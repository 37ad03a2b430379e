"""Pins of the float64 gradient oracle (``oracle/attn_grad_oracle.c``).

The pages give no gradient formulas, only what a backward pass keeps and
rebuilds ("FlashAttention: The Matrix You Never Have to Write Down", section
"The forward pass is only half of it").  So the gradient oracle is pinned
to things other than its own formulas:

* central finite differences of the forward oracle's scalar sum(dO * O),
  element by element, on tiny square and non-square, causal and unmasked
  shapes — this fixes every term of all three gradients;
* torch float64 autograd through softmax and matmul (a library routine);
* closed forms: one key (dQ = dK = 0, dV = dO); identical keys (dQ = 0);
  zero keys (uniform weights, dV in closed form); the key-sum of dK is zero
  (every softmax-Jacobian row sums to zero); D equals dO . O of the forward
  oracle.

Each pin takes a loaded oracle library and raises AssertionError on a
mismatch.
"""
import math

import numpy as np

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _loss(lib, q, k, v, g, causal, scale):
    o, _ = oracle.attention(q, k, v, causal=causal, scale=scale, lib=lib)
    return float((o * g).sum())


def pin_grad_finite_differences(lib):
    """Every gradient element against a central difference of sum(dO * O)."""
    h = 1e-5
    for (tq, tk, d, dv, causal, seed) in [(5, 5, 3, 4, False, 1), (5, 5, 3, 4, True, 2),
                                          (4, 6, 2, 3, True, 3), (6, 3, 3, 2, False, 4)]:
        r = _rng(seed)
        q, k = r.standard_normal((tq, d)), r.standard_normal((tk, d))
        v, g = r.standard_normal((tk, dv)), r.standard_normal((tq, dv))
        scale = 0.7
        dq, dk, dvv = oracle.attention_grad(q, k, v, g, causal=causal, scale=scale, lib=lib)
        for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                args_p[name], args_m[name] = xp, xm
                fd = (_loss(lib, args_p["q"], args_p["k"], args_p["v"], g, causal, scale) -
                      _loss(lib, args_m["q"], args_m["k"], args_m["v"], g, causal, scale)) / (2 * h)
                assert abs(fd - grad[idx]) <= 1e-7 * (1.0 + abs(fd)), \
                    (name, idx, fd, grad[idx], tq, tk, causal)


def pin_grad_vs_torch(lib):
    """torch float64 autograd of softmax(scale Q K^T, masked) V."""
    import torch
    for (b, tq, tk, d, dv, causal, seed) in [(3, 17, 17, 8, 8, False, 5), (2, 33, 33, 16, 16, True, 6),
                                             (2, 9, 21, 4, 5, True, 7), (1, 20, 7, 6, 3, False, 8)]:
        r = _rng(seed)
        q, k = r.standard_normal((b, tq, d)), r.standard_normal((b, tk, d))
        v, g = r.standard_normal((b, tk, dv)), r.standard_normal((b, tq, dv))
        scale = 1.0 / math.sqrt(d)
        tq_, tk_, tv_ = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        s = scale * tq_ @ tk_.transpose(-1, -2)
        if causal:
            mask = torch.ones(tq, tk, dtype=torch.bool).tril()
            s = s.masked_fill(~mask, float("-inf"))
        o = torch.softmax(s, dim=-1) @ tv_
        (o * torch.tensor(g)).sum().backward()
        dq, dk, dvv = oracle.attention_grad(q, k, v, g, causal=causal, scale=scale, lib=lib)
        for mine, ref in ((dq, tq_.grad), (dk, tk_.grad), (dvv, tv_.grad)):
            assert np.abs(mine - ref.numpy()).max() <= 1e-10 * (1 + np.abs(ref.numpy()).max())


def pin_grad_single_key(lib):
    """One key: softmax weight 1, so dV = dO and dQ = dK = 0."""
    r = _rng(9)
    q, k = r.standard_normal((1, 1, 8)), r.standard_normal((1, 1, 8))
    v, g = r.standard_normal((1, 1, 8)), r.standard_normal((1, 1, 8))
    for causal in (False, True):
        dq, dk, dvv = oracle.attention_grad(q, k, v, g, causal=causal, lib=lib)
        assert np.abs(dq).max() <= 1e-14 and np.abs(dk).max() <= 1e-14
        assert np.abs(dvv - g).max() <= 1e-14


def pin_grad_key_sum_zero(lib):
    """sum_j dK[j] = scale * sum_i (sum_j dS[i][j]) Q[i] = 0: Jacobian rows sum to zero."""
    r = _rng(10)
    for causal in (False, True):
        q, k = r.standard_normal((2, 40, 16)), r.standard_normal((2, 40, 16))
        v, g = r.standard_normal((2, 40, 16)), r.standard_normal((2, 40, 16))
        dq, dk, dvv = oracle.attention_grad(q, k, v, g, causal=causal, lib=lib)
        assert np.abs(dk.sum(axis=1)).max() <= 1e-12 * (1 + np.abs(dk).max())
        assert np.abs(dk).max() > 1e-3   # and dK itself is not trivially zero


def pin_grad_equal_keys(lib):
    """Identical keys: dQ[i] = scale * (sum_j dS[i][j]) k = 0."""
    r = _rng(11)
    q = r.standard_normal((1, 12, 8))
    k = np.repeat(r.standard_normal((1, 1, 8)), 12, axis=1)
    v, g = r.standard_normal((1, 12, 8)), r.standard_normal((1, 12, 8))
    for causal in (False, True):
        dq, _, _ = oracle.attention_grad(q, k, v, g, causal=causal, lib=lib)
        assert np.abs(dq).max() <= 1e-13


def pin_grad_uniform(lib):
    """K = 0: weights 1/n_i over the visible keys, so dV[j] = sum_{i sees j} dO[i] / n_i."""
    r = _rng(12)
    n, dv = 10, 5
    q = r.standard_normal((1, n, 4))
    k = np.zeros((1, n, 4))
    v, g = r.standard_normal((1, n, dv)), r.standard_normal((1, n, dv))
    for causal in (False, True):
        _, _, dvv = oracle.attention_grad(q, k, v, g, causal=causal, lib=lib)
        want = np.zeros((n, dv))
        for i in range(n):
            nvis = i + 1 if causal else n
            for j in range(nvis):
                want[j] += g[0, i] / nvis
        assert np.abs(dvv[0] - want).max() <= 1e-13


def pin_grad_rows_api(lib):
    """Row-selected passes agree with whole heads; D equals dO . O of the forward oracle."""
    r = _rng(13)
    n, d, dv = 50, 8, 6
    q, k = r.standard_normal((n, d)), r.standard_normal((n, d))
    v, g = r.standard_normal((n, dv)), r.standard_normal((n, dv))
    for causal in (False, True):
        dq, dk, dvv = oracle.attention_grad(q, k, v, g, causal=causal, scale=0.4, lib=lib)
        rows = np.arange(n)
        dq_r, lse, delta = oracle.grad_query_rows(q, g, rows, k, v, causal=causal, scale=0.4, lib=lib)
        o, lse_f = oracle.attention(q, k, v, causal=causal, scale=0.4, lib=lib)
        assert np.abs(delta - (o * g).sum(axis=1)).max() <= 1e-12
        assert np.abs(lse - lse_f).max() <= 1e-12
        assert np.abs(dq_r - dq).max() <= 1e-13
        sel = np.array([0, 7, 31, 49])
        dk_r, dv_r = oracle.grad_key_rows(k[sel], v[sel], sel, q, g, lse, delta, causal=causal,
                                          scale=0.4, lib=lib)
        assert np.abs(dk_r - dk[sel]).max() <= 1e-13
        assert np.abs(dv_r - dvv[sel]).max() <= 1e-13


def pin_grad_rows_lower_right_vs_torch(lib):
    """The row passes with bottom-right positions (queries at i + Nk - Nq,
    keys at j, or equivalently keys at j - (Nk - Nq) against queries at i,
    the form the kv and packed backward tests use) against torch float64
    autograd through SDPA with its lower-right causal bias, Nq <= Nk."""
    import torch
    from torch.nn.attention.bias import causal_lower_right
    F = torch.nn.functional
    for (tq, tk, d, dv, seed) in [(5, 23, 8, 8, 31), (12, 12, 4, 6, 32), (1, 9, 8, 3, 33)]:
        r = _rng(seed)
        q, k = r.standard_normal((tq, d)), r.standard_normal((tk, d))
        v, g = r.standard_normal((tk, dv)), r.standard_normal((tq, dv))
        scale = 1.0 / math.sqrt(d)
        tq_, tk_, tv_ = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        o = F.scaled_dot_product_attention(tq_[None, None], tk_[None, None], tv_[None, None],
                                           attn_mask=causal_lower_right(tq, tk), scale=scale)[0, 0]
        (o * torch.tensor(g)).sum().backward()
        off = tk - tq
        dq, lse, delta = oracle.grad_query_rows(q, g, np.arange(tq) + off, k, v, causal=True,
                                                scale=scale, lib=lib)
        dk, dvv = oracle.grad_key_rows(k, v, np.arange(tk) - off, q, g, lse, delta, causal=True,
                                       scale=scale, lib=lib)
        for mine, ref in ((dq, tq_.grad), (dk, tk_.grad), (dvv, tv_.grad)):
            assert np.abs(mine - ref.numpy()).max() <= 1e-10 * (1 + np.abs(ref.numpy()).max())


ALL_GRAD_PINS = [pin_grad_finite_differences, pin_grad_vs_torch, pin_grad_single_key,
                 pin_grad_key_sum_zero, pin_grad_equal_keys, pin_grad_uniform,
                 pin_grad_rows_api, pin_grad_rows_lower_right_vs_torch]
