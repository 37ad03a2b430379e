"""Pins for the float64 oracle: facts fixed by the pages or by mathematics.

Each ``pin_*`` takes a loaded oracle library and raises AssertionError when
the oracle disagrees.  They are collected here (not inside the test module)
so that ``test_oracle_mutants.py`` can run the same pins against copies of the
oracle with a planted mistake and check that every such mistake is caught.
"""
import math
import os

import numpy as np
import torch

import oracle
from oracle import online_model

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Parse a ``key = value`` fixture; values stay strings."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out[key] = val
    return out


def _num(tok):
    tok = tok.strip()
    if tok == "ln2":
        return math.log(2.0)
    if tok in ("-inf", "inf"):
        return float(tok)
    return float(tok)


def _nums(s):
    return [_num(t) for t in s.split()]


def _round_eq(value, printed, digits):
    return round(float(value), int(digits)) == round(float(printed), int(digits))


def _rng(seed):
    return np.random.default_rng(seed)


# --- the pages' worked examples ------------------------------------------------

def pin_four_numbers(lib):
    """Four scores in two blocks: sums 1.3679 then 1.000504 (pages' printout)."""
    g = read_golden("four_numbers.txt")
    scores = _nums(g["block1"]) + _nums(g["block2"])
    # d = 1, q = 1, scale = 1: the scores are the keys themselves.
    q = np.ones((1, 1))
    k = np.array(scores).reshape(-1, 1)
    v = np.zeros((len(scores), 1))
    _, lse = oracle.attention(q, k, v, scale=1.0, lib=lib)
    dense_sum = math.exp(lse[0] - max(scores))       # sum of exp(x - max)
    assert _round_eq(dense_sum, g["dense_sum"], g["dense_sum_digits"]), dense_sum
    # The same quantity by the one-pass recurrence, block size 2.
    lse2 = online_model.streaming_lse(scores, block=2)
    assert abs(lse2 - lse[0]) < 1e-14
    b1 = np.array(_nums(g["block1"]))
    m1 = b1.max()
    assert m1 == float(g["after_block1_max"])
    assert _round_eq(np.exp(b1 - m1).sum(), g["after_block1_sum"],
                     g["after_block1_sum_digits"])
    alpha = math.exp(m1 - float(g["block2_max"]))
    assert abs(alpha / float(g["alpha"]) - 1) < float(g["alpha_rel"])
    trace = []
    online_model.online_attention(q, k, v, block_k=2, scale=1.0, trace=trace)
    assert _round_eq(trace[-1][4], g["after_block2_sum"], g["after_block2_sum_digits"])
    assert abs(trace[-1][3] - alpha) < 1e-18


def pin_two_block(lib):
    """Scores 0,0,ln2,ln2 with values 0,0,10,10 give 20/3, not 5."""
    g = read_golden("two_block.txt")
    s = np.array(_nums(g["scores"]))
    vals = np.array(_nums(g["values"])).reshape(-1, 1)
    q = np.ones((1, 1))
    k = s.reshape(-1, 1)
    o, lse = oracle.attention(q, k, vals, scale=1.0, lib=lib)
    want = float(g["output_num"]) / float(g["output_den"])
    assert abs(o[0, 0] - want) < 1e-13, o
    assert abs(o[0, 0] - float(g["naive_block_mean"])) > 1.0
    # LSE = ln(1 + 1 + 2 + 2) = ln 6.
    assert abs(lse[0] - math.log(6.0)) < 1e-14
    trace = []
    o2, _ = online_model.online_attention(q, k, vals, block_k=2, scale=1.0, trace=trace)
    assert abs(o2[0, 0] - want) < 1e-13
    _, _, m1, _, l1 = trace[0]
    _, _, m2, a2, l2 = trace[1]
    assert m1 == _num(g["block1_max"]) and l1 == float(g["block1_sum"])
    assert abs(m2 - _num(g["block2_max"])) < 1e-15
    assert abs(a2 - float(g["block1_rescale"])) < 1e-15
    assert abs(l2 - float(g["combined_denominator"])) < 1e-14


def pin_late_max(lib):
    """Max in the final key tile: prints 4.0000000."""
    g = read_golden("late_max.txt")
    q = np.array([[float(g["q"])]])
    k = np.array(_nums(g["keys"])).reshape(-1, 1)
    v = np.array(_nums(g["values"])).reshape(-1, 1)
    o, lse = oracle.attention(q, k, v, lib=lib)          # scale 1/sqrt(1)
    assert f"{o[0, 0]:.{g['output_digits']}f}" == g["output"], o
    e = math.exp(-20.0)
    exact = (1 * e + 2 * e + 3 * e + 4) / (3 * e + 1)
    assert abs(o[0, 0] - exact) < 1e-15
    assert abs(lse[0] - (20.0 + math.log(1 + 3 * e))) < 1e-13
    o2, _ = online_model.online_attention(q, k, v, block_k=int(g["block_k"]))
    assert abs(o2[0, 0] - exact) < 1e-15


def pin_empty_keys(lib):
    """No keys: O = 0 and LSE = -inf, by policy."""
    g = read_golden("empty_keys.txt")
    tq, d, tk, dv = (int(g[x]) for x in ("tq", "d", "tk", "dv"))
    q = _rng(5).standard_normal((tq, d))
    o, lse = oracle.attention(q, np.zeros((tk, d)), np.zeros((tk, dv)), lib=lib)
    assert o.shape == (tq, dv) and np.all(o == float(g["output"]))
    assert np.all(np.isneginf(lse))


# --- invariants and special cases ---------------------------------------------

def pin_rows_sum_to_one(lib):
    """V = all ones gives O = 1 (the weights of a row sum to one)."""
    r = _rng(11)
    for causal in (False, True):
        q = r.standard_normal((2, 37, 16)) * 3
        k = r.standard_normal((2, 37, 16))
        v = np.ones((2, 37, 5))
        o, _ = oracle.attention(q, k, v, causal=causal, lib=lib)
        assert np.max(np.abs(o - 1.0)) < 1e-13


def pin_equal_scores(lib):
    """K = 0: every visible score is 0, O = mean of visible V, LSE = ln(count)."""
    r = _rng(12)
    n, d, dv = 29, 8, 6
    q = r.standard_normal((n, d))
    k = np.zeros((n, d))
    v = r.standard_normal((n, dv))
    o, lse = oracle.attention(q, k, v, lib=lib)
    assert np.max(np.abs(o - v.mean(axis=0))) < 1e-13
    assert np.max(np.abs(lse - math.log(n))) < 1e-13
    o, lse = oracle.attention(q, k, v, causal=True, lib=lib)
    for i in range(n):
        assert np.max(np.abs(o[i] - v[:i + 1].mean(axis=0))) < 1e-13
        assert abs(lse[i] - math.log(i + 1)) < 1e-13


def pin_single_key(lib):
    """N = 1: O = V and LSE = scale * q.k."""
    r = _rng(13)
    q, k, v = (r.standard_normal((3, 1, 7)) for _ in range(3))
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal=causal, scale=0.3, lib=lib)
        assert np.max(np.abs(o - v)) < 1e-15
        want = 0.3 * np.einsum("hid,hid->hi", q, k)
        assert np.max(np.abs(lse - want)) < 1e-14


def pin_causal_row0(lib):
    """Causal row 0 sees only key 0: O[0] = V[0]; and query i always sees key i."""
    r = _rng(14)
    q, k = r.standard_normal((40, 8)) * 5, r.standard_normal((40, 8))
    v = r.standard_normal((40, 3))
    o, lse = oracle.attention(q, k, v, causal=True, lib=lib)
    assert np.max(np.abs(o[0] - v[0])) < 1e-15
    assert abs(lse[0] - q[0] @ k[0] / math.sqrt(8)) < 1e-13
    # the last row sees everything, like the unmasked row
    o2, lse2 = oracle.attention(q, k, v, causal=False, lib=lib)
    assert np.max(np.abs(o[-1] - o2[-1])) < 1e-14 and abs(lse[-1] - lse2[-1]) < 1e-13


def pin_permutation(lib):
    """Unmasked attention is invariant to a joint reordering of the K/V pairs."""
    r = _rng(3)
    q, k, v = r.standard_normal((96, 32)), r.standard_normal((96, 32)), r.standard_normal((96, 24))
    perm = r.permutation(96)
    o1, l1 = oracle.attention(q, k, v, lib=lib)
    o2, l2 = oracle.attention(q, k[perm], v[perm], lib=lib)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def pin_score_shift(lib):
    """Adding c to every score leaves O unchanged and adds c to LSE."""
    r = _rng(15)
    n, d = 33, 12
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, 4))
    c = 7.25
    # an extra column: q gets c/scale, k gets 1  ->  every score grows by c
    scale = 0.5
    qa = np.concatenate([q, np.full((n, 1), c / scale)], axis=1)
    ka = np.concatenate([k, np.ones((n, 1))], axis=1)
    for causal in (False, True):
        o1, l1 = oracle.attention(q, k, v, causal=causal, scale=scale, lib=lib)
        o2, l2 = oracle.attention(qa, ka, v, causal=causal, scale=scale, lib=lib)
        assert np.max(np.abs(o1 - o2)) < 1e-12
        assert np.max(np.abs(l2 - l1 - c)) < 1e-12


def pin_large_scores(lib):
    """Scores in the thousands stay finite: O -> V at the argmax, LSE -> max."""
    r = _rng(16)
    n, d = 20, 4
    k = r.standard_normal((n, d))
    q = k[7:8] * 1000.0                    # the score with key 7 dominates
    v = r.standard_normal((n, 3))
    o, lse = oracle.attention(q, k, v, scale=1.0, lib=lib)
    s = (q @ k.T)[0]
    assert np.all(np.isfinite(o)) and np.isfinite(lse[0])
    top = int(np.argmax(s))
    gap = s[top] - np.partition(s, -2)[-2]
    assert gap > 50
    assert np.max(np.abs(o[0] - v[top])) < 1e-12
    assert abs(lse[0] - s[top]) < 1e-9 * abs(s[top])


def pin_value_affine(lib):
    """O is a convex blend of V: O(a V + b) = a O(V) + b."""
    r = _rng(17)
    q, k, v = r.standard_normal((25, 9)), r.standard_normal((25, 9)), r.standard_normal((25, 9))
    for causal in (False, True):
        o1, _ = oracle.attention(q, k, v, causal=causal, lib=lib)
        o2, _ = oracle.attention(q, k, 2.5 * v - 1.25, causal=causal, lib=lib)
        assert np.max(np.abs(o2 - (2.5 * o1 - 1.25))) < 1e-12


def pin_vs_torch(lib):
    """Small shapes against torch's float64 CPU softmax and SDPA (incl. non-square causal)."""
    gen = torch.Generator().manual_seed(21)
    shapes = [(64, 64, 16, 16), (100, 100, 32, 32), (128, 96, 64, 24), (37, 53, 8, 11)]
    for tq, tk, d, dv in shapes:
        q = torch.randn(tq, d, generator=gen, dtype=torch.float64)
        k = torch.randn(tk, d, generator=gen, dtype=torch.float64)
        v = torch.randn(tk, dv, generator=gen, dtype=torch.float64)
        s = (q @ k.T) / math.sqrt(d)
        want_o = torch.softmax(s, -1) @ v
        want_l = torch.logsumexp(s, -1)
        o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), lib=lib)
        assert np.max(np.abs(o - want_o.numpy())) < 1e-12
        assert np.max(np.abs(lse - want_l.numpy())) < 1e-12
    F = torch.nn.functional
    for tq, tk in [(3, 7), (7, 3), (1, 10), (10, 1), (64, 64)]:
        q = torch.randn(tq, 8, generator=gen, dtype=torch.float64)
        k = torch.randn(tk, 8, generator=gen, dtype=torch.float64)
        v = torch.randn(tk, 5, generator=gen, dtype=torch.float64)
        want = F.scaled_dot_product_attention(q[None, None], k[None, None],
                                              v[None, None], is_causal=True)[0, 0]
        o, _ = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=True, lib=lib)
        assert np.max(np.abs(o - want.numpy())) < 1e-12


def pin_rows_lower_right_vs_torch(lib):
    """Queries at positions shifted by the key/query length difference (the
    bottom-right causal alignment of a chunk after a cache) against torch's
    float64 SDPA with its lower-right causal bias; with more queries than
    keys the first rows see nothing and must come back O = 0, LSE = -inf."""
    from torch.nn.attention.bias import causal_lower_right
    import warnings
    F = torch.nn.functional
    gen = torch.Generator().manual_seed(23)
    for tq, tk in [(3, 7), (5, 40), (1, 17), (16, 16), (9, 4)]:
        q = torch.randn(tq, 8, generator=gen, dtype=torch.float64)
        k = torch.randn(tk, 8, generator=gen, dtype=torch.float64)
        v = torch.randn(tk, 5, generator=gen, dtype=torch.float64)
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            bias = causal_lower_right(tq, tk)
            want = F.scaled_dot_product_attention(q[None, None], k[None, None], v[None, None],
                                                  attn_mask=bias)[0, 0].numpy()
        pos = np.arange(tq, dtype=np.int64) + (tk - tq)
        o, lse = oracle.attention_rows(q.numpy(), pos, k.numpy(), v.numpy(), causal=True, lib=lib)
        seen = pos >= 0
        assert np.max(np.abs(o[seen] - want[seen])) < 1e-12, (tq, tk)
        s = (q @ k.T).numpy() / math.sqrt(8)
        mask = np.arange(tk)[None, :] <= pos[:, None]
        want_l = np.array([np.log(np.sum(np.exp(s[i][mask[i]] - s[i][mask[i]].max())))
                           + s[i][mask[i]].max() for i in range(tq) if seen[i]])
        assert np.max(np.abs(lse[seen] - want_l)) < 1e-12
        assert np.all(o[~seen] == 0.0) and np.all(np.isneginf(lse[~seen]))


def pin_online_model(lib):
    """Online fold over key blocks vs the one-shot oracle, ragged blocks."""
    r = _rng(22)
    shapes = [(64, 64, 16, 16), (100, 100, 32, 32), (128, 96, 64, 24), (37, 53, 8, 11)]
    for tq, tk, d, dv in shapes:
        for causal in ([False, True] if tq == tk else [False]):
            for bk in (32, 64, 13, 7):
                q = r.standard_normal((tq, d)) * 2
                k, v = r.standard_normal((tk, d)), r.standard_normal((tk, dv))
                o1, l1 = online_model.online_attention(q, k, v, causal, bk)
                o2, l2 = oracle.attention(q, k, v, causal=causal, lib=lib)
                assert np.max(np.abs(o1 - o2)) < 1e-12, (tq, tk, causal, bk)
                assert np.max(np.abs(l1 - l2)) < 1e-12


def pin_rows_api(lib):
    """Sampled rows agree with whole heads, at any positions and order."""
    r = _rng(23)
    n, d = 70, 16
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal=causal, lib=lib)
        rows = np.array([69, 0, 13, 64, 1, 35])
        o2, l2 = oracle.attention_rows(q[rows], rows, k, v, causal=causal, lib=lib)
        assert np.max(np.abs(o2 - o[rows])) == 0.0 and np.max(np.abs(l2 - lse[rows])) == 0.0


ALL_PINS = [pin_rows_lower_right_vs_torch, pin_four_numbers, pin_two_block, pin_late_max, pin_empty_keys,
            pin_rows_sum_to_one, pin_equal_scores, pin_single_key, pin_causal_row0,
            pin_permutation, pin_score_shift, pin_large_scores, pin_value_affine,
            pin_vs_torch, pin_online_model, pin_rows_api]
