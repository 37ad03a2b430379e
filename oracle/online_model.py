"""Online-softmax model in float64.  TEST INFRASTRUCTURE ONLY.

A second derivation of attention, independent of the one-shot definition in
``attn_oracle.c``: it never holds more than one block of a score row, and it
reaches the result through the combining identity that the online softmax
rests on ("FlashAttention: The Matrix You Never Have to Write Down", section
"The identity: you can fix what you already wrote", for the running maximum
and sum; section "From softmax to attention: rescale the output too", for
the output vector that is rescaled by the same factor).

The model is built on summaries.  A piece of one score row s with values v
is summarised by three numbers' worth of state,

    m = max s,   l = sum exp(s - m),   o = sum exp(s - m) * v,

and the summaries of two disjoint pieces give the summary of their union
exactly: with M the larger maximum, each side is scaled by exp(its m - M)
and the scaled sums are added.  An empty piece (no entry, or only -inf
entries) has m = -inf and l = 0 and carries no weight, so combining with it
never evaluates exp(-inf - (-inf)).  At the end the row's output is o / l
and its log-sum-exp m + ln l; a row with nothing visible gets O = 0 and
L = -inf (section "Check it", the empty-key policy).

``online_attention`` folds the key blocks of each query row into a running
summary, left to right, one row at a time; with causal masking row i sees
keys 0 .. i (upper-left alignment, section "Build it", its note on causal
alignment), so its last block is cut at the diagonal.  numpy is used only
as a vector library (a block's scores, exp, max, a weighted sum).
"""
import math

import numpy as np


def summarise(s, v=None):
    """Summary (m, l, o) of scores ``s`` (1-D) with value rows ``v``.

    ``o`` is None when ``v`` is None (log-sum-exp only).
    """
    s = np.asarray(s, dtype=np.float64)
    dv = None if v is None else np.asarray(v).shape[1]
    m = float(s.max()) if s.size else -math.inf
    if m == -math.inf:
        return -math.inf, 0.0, (None if v is None else np.zeros(dv))
    w = np.exp(s - m)
    return m, float(w.sum()), (None if v is None else w @ np.asarray(v, dtype=np.float64))


def combine(a, b):
    """Summary of the union of two disjoint pieces, and the factor that
    multiplied ``a``'s sums (0 when ``a`` was empty)."""
    ma, la, oa = a
    mb, lb, ob = b
    if la == 0.0:
        return b, 0.0
    if lb == 0.0:
        return a, 1.0
    M = max(ma, mb)
    fa, fb = math.exp(ma - M), math.exp(mb - M)
    o = None if oa is None else oa * fa + ob * fb
    return (M, la * fa + lb * fb, o), fa


def streaming_lse(x, block=5):
    """log(sum(exp(x))) by folding block summaries left to right."""
    x = np.asarray(x, dtype=np.float64).ravel()
    if block < 1:
        raise ValueError("block size must be positive")
    state = (-math.inf, 0.0, None)
    for start in range(0, x.size, block):
        state, _ = combine(state, summarise(x[start:start + block]))
    m, l, _ = state
    return m + math.log(l) if l > 0.0 else -math.inf


def online_attention(Q, K, V, causal=False, block_k=32, scale=None, trace=None):
    """Attention of one head by the online fold, in float64.

    Q: (Tq, d), K: (Tk, d), V: (Tk, dv) -> O: (Tq, dv), L: (Tq,).
    ``scale`` defaults to 1/sqrt(d); key blocks start at multiples of
    ``block_k``.  When ``trace`` is a list, every fold step appends
    (row, key block start, m, factor applied to the old sums, l) so a test
    can read the intermediate values of a worked example.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if Q.ndim != 2 or K.ndim != 2 or V.ndim != 2:
        raise ValueError("Q, K, V must be rank 2 (one head)")
    if K.shape[1] != Q.shape[1]:
        raise ValueError("Q and K widths differ")
    if V.shape[0] != K.shape[0]:
        raise ValueError("K and V lengths differ")
    if Q.shape[1] == 0:
        raise ValueError("width must be positive")
    if block_k < 1:
        raise ValueError("block size must be positive")
    Tq, d = Q.shape
    Tk, dv = K.shape[0], V.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)

    O = np.zeros((Tq, dv))
    L = np.full((Tq,), -math.inf)
    for i in range(Tq):
        visible = min(Tk, i + 1) if causal else Tk
        state = (-math.inf, 0.0, np.zeros(dv))
        for j in range(0, visible, block_k):
            stop = min(j + block_k, visible)
            s = (K[j:stop] @ Q[i]) * scale
            state, factor = combine(state, summarise(s, V[j:stop]))
            if trace is not None:
                trace.append((i, j, state[0], factor, state[1]))
        m, l, o = state
        if l > 0.0:
            O[i] = o / l
            L[i] = m + math.log(l)
    return O, L
