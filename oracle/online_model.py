"""Block-wise online-softmax model in float64.  TEST INFRASTRUCTURE ONLY.

This is the second, independent derivation of attention that the oracle is
pinned against: it never forms a whole score row, and reaches the result
through the running-maximum / running-sum recurrence instead of the one-shot
definition in ``attn_oracle.c``.  It follows the steps and notation of
"FlashAttention: The Matrix You Never Have to Write Down":

* ``streaming_lse`` — section "The identity: you can fix what you already
  wrote": one pass over blocks holding (m, l); a block whose entries are all
  -inf is skipped, the first rescale factor is forced to 0 instead of
  computing exp(-inf - (-inf)), and an input with nothing finite gives -inf.
* ``online_attention`` — section "From softmax to attention: rescale the
  output too" (the m_new / alpha / P / l / O equations) with the loop
  structure of section "Build it": query blocks outside, key/value blocks
  inside, a causal query block stops at the first key block that lies wholly
  in its future, the block that straddles the diagonal is masked per element
  (key position > query position), and O is divided by l once at the end.
  An empty key sequence returns O = 0 and L = -inf (section "Check it").

numpy is used only as a vector library (a block matmul, exp, max); there is
no blocking or reordering beyond what the recurrence states.
"""
import math

import numpy as np


def streaming_lse(x, block=7):
    """log(sum(exp(x))) in one pass over blocks of ``block`` entries."""
    x = np.asarray(x, dtype=np.float64).ravel()
    m, l = -math.inf, 0.0
    for start in range(0, x.size, block):
        blk = x[start:start + block]
        bmax = float(blk.max())
        if bmax == -math.inf:
            continue                      # contributes nothing
        m_new = max(m, bmax)
        alpha = 0.0 if m == -math.inf else math.exp(m - m_new)
        l = l * alpha + float(np.exp(blk - m_new).sum())
        m = m_new
    return -math.inf if l == 0.0 else m + math.log(l)


def online_attention(Q, K, V, causal=False, block_q=32, block_k=32, scale=None,
                     trace=None):
    """Tiled attention for one head by the online recurrence, in float64.

    Q: (Tq, d), K: (Tk, d), V: (Tk, dv) -> O: (Tq, dv), L: (Tq,).
    ``scale`` defaults to 1/sqrt(d).  When ``trace`` is a list, every update
    appends (query block start, key block start, m_new, alpha, l) so a test
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
    if block_q < 1 or block_k < 1:
        raise ValueError("block sizes must be positive")
    Tq, d = Q.shape
    Tk, dv = K.shape[0], V.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if Tk == 0:
        return np.zeros((Tq, dv)), np.full((Tq,), -math.inf)

    O = np.zeros((Tq, dv))
    L = np.zeros((Tq,))
    for i in range(0, Tq, block_q):
        nq = min(block_q, Tq - i)
        Qi = Q[i:i + nq]
        Oi = np.zeros((nq, dv))            # unnormalised output so far
        mi = np.full((nq,), -math.inf)     # running maximum
        li = np.zeros((nq,))               # running sum of exponentials
        for j in range(0, Tk, block_k):
            if causal and j > i + nq - 1:
                break                      # this and every later block is future
            nk = min(block_k, Tk - j)
            S = (Qi @ K[j:j + nk].T) * scale
            if causal:
                qpos = np.arange(i, i + nq)[:, None]
                kpos = np.arange(j, j + nk)[None, :]
                S = np.where(kpos > qpos, -math.inf, S)
            m_new = np.maximum(mi, S.max(axis=1))
            with np.errstate(invalid="ignore"):
                alpha = np.where(np.isneginf(mi), 0.0, np.exp(mi - m_new))
            P = np.exp(S - m_new[:, None])
            li = li * alpha + P.sum(axis=1)
            Oi = Oi * alpha[:, None] + P @ V[j:j + nk]
            mi = m_new
            if trace is not None:
                trace.append((i, j, m_new.copy(), alpha.copy(), li.copy()))
        O[i:i + nq] = Oi / li[:, None]
        L[i:i + nq] = mi + np.log(li)
    return O, L
