"""Float64 CPU oracle for exact attention.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never import, link or call it, and it imports nothing from them.

* ``attention`` / ``attention_rows`` — the plain definition (scores, row max,
  exp-sum, V blend, logsumexp) in C, ``attn_oracle.c``.
* ``attention_grad`` / ``grad_query_rows`` / ``grad_key_rows`` — the
  gradients of that definition with respect to Q, K and V (chain rule through
  the softmax) in C, ``attn_grad_oracle.c``.
* ``attention_dropout`` / ``attention_dropout_grad`` / ``dropout_mask`` /
  ``philox4x32_10`` — attention with dropout on the weights, its gradients,
  the keep mask and the counter-based generator it is drawn from, in C,
  ``attn_dropout_oracle.c``.
* ``online_model`` — the online softmax in numpy, as a left-to-right fold
  of block summaries (maximum, exp-sum, weighted values) combined by the
  rescale identity: the second derivation the C code is pinned against.

``build()`` compiles the C files with gcc (OpenMP over rows) into
``oracle/_build/liboracle.so``; the first call to ``attention`` builds it if
it is missing.
"""
import ctypes
import math
import os
import subprocess

import numpy as np

from . import online_model  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_GRAD_SRC = os.path.join(_HERE, "attn_grad_oracle.c")
_DROP_SRC = os.path.join(_HERE, "attn_dropout_oracle.c")
SOURCES = (_SRC, _GRAD_SRC, _DROP_SRC)
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None


def compile_oracle(src=SOURCES, out=_LIB_PATH, extra_flags=()):
    """Compile oracle source file(s) into a shared library; returns the path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    srcs = [src] if isinstance(src, (str, os.PathLike)) else list(src)
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99", *extra_flags,
           *srcs, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build():
    """Compile the oracle (always rebuilds)."""
    global _lib
    _lib = None
    compile_oracle()
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_attention_rows.argtypes = [i64, i64, i64, p, p, i64, p, p,
                                          ctypes.c_int, ctypes.c_double, p, p]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [i64, i64, i64, i64, i64, p, p, p,
                                     ctypes.c_int, ctypes.c_double, p, p]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    if hasattr(lib, "oracle_attention_grad"):   # a forward-only build has none
        i32, f64 = ctypes.c_int, ctypes.c_double
        lib.oracle_attention_grad.argtypes = [i64, i64, i64, i64, i64, p, p, p, p, i32, f64,
                                              p, p, p]
        lib.oracle_attention_grad.restype = i32
        lib.oracle_grad_query_rows.argtypes = [i64, i64, i64, p, p, i64, p, p, p, i32, f64,
                                               p, p, p]
        lib.oracle_grad_query_rows.restype = i32
        lib.oracle_grad_key_rows.argtypes = [i64, i64, i64, p, p, p, p, i64, p, p, p, i32,
                                             f64, p, p]
        lib.oracle_grad_key_rows.restype = i32
    if hasattr(lib, "oracle_attention_dropout"):
        i32, f64, u32, u64 = ctypes.c_int, ctypes.c_double, ctypes.c_uint32, ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [p, p, p]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_dropout_mask.argtypes = [i64, i64, i64, u64, u32, i32, p]
        lib.oracle_dropout_mask.restype = i32
        lib.oracle_attention_dropout.argtypes = [i64, i64, i64, i64, i64, p, p, p, i32, i64,
                                                 f64, u64, u32, i32, p, p]
        lib.oracle_attention_dropout.restype = i32
        lib.oracle_attention_dropout_grad.argtypes = [i64, i64, i64, i64, i64, p, p, p, p, i32,
                                                      i64, f64, u64, u32, i32, p, p, p]
        lib.oracle_attention_dropout_grad.restype = i32
    return lib


def load(path=None):
    """The compiled oracle (building it first when it is missing)."""
    global _lib
    if path is not None:
        return _bind(path)
    if _lib is None:
        if not os.path.exists(_LIB_PATH) or any(
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(f) for f in SOURCES):
            compile_oracle()
        _lib = _bind(_LIB_PATH)
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


def attention(q, k, v, causal=False, scale=None, lib=None):
    """Exact attention over the last two axes, in float64.

    q [..., Tq, d], k [..., Tk, d], v [..., Tk, dv] (any leading batch/head
    axes, identical for all three) -> (o [..., Tq, dv], lse [..., Tq]).
    Query i sits at position i (upper-left causal alignment).  ``scale``
    defaults to 1/sqrt(d).
    """
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead = q.shape[:-2]
    if k.shape[:-2] != lead or v.shape[:-2] != lead:
        raise ValueError("q, k, v leading axes differ")
    tq, d = q.shape[-2:]
    tk, dv = v.shape[-2:]
    if k.shape[-1] != d or k.shape[-2] != tk:
        raise ValueError("k shape does not match q/v")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bh = int(np.prod(lead)) if lead else 1
    o = np.zeros(lead + (tq, dv))
    lse = np.zeros(lead + (tq,))
    rc = lib.oracle_attention(bh, tq, tk, d, dv, _ptr(q), _ptr(k), _ptr(v),
                              int(bool(causal)), float(scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_attention failed ({rc})")
    return o, lse


def attention_rows(q_rows, q_pos, k, v, causal=False, scale=None, lib=None):
    """Exact attention for selected query rows of ONE head.

    q_rows [R, d] with absolute positions q_pos [R]; k [Tk, d]; v [Tk, dv]
    -> (o [R, dv], lse [R]).
    """
    lib = lib or load()
    q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
    pos = np.ascontiguousarray(np.asarray(q_pos, dtype=np.int64))
    r, d = q_rows.shape
    tk, dv = v.shape
    if pos.shape != (r,) or k.shape != (tk, d):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((r, dv))
    lse = np.zeros((r,))
    rc = lib.oracle_attention_rows(tk, d, dv, _ptr(k), _ptr(v), r, _ptr(q_rows),
                                   _ptr(pos), int(bool(causal)), float(scale),
                                   _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed ({rc})")
    return o, lse


def num_threads(lib=None):
    """OpenMP threads the oracle runs rows on."""
    return int((lib or load()).oracle_num_threads())


def attention_grad(q, k, v, dout, causal=False, scale=None, lib=None):
    """Gradients of exact attention over the last two axes, in float64.

    q [..., Tq, d], k [..., Tk, d], v [..., Tk, dv], dout [..., Tq, dv] ->
    (dq, dk, dv) of the scalar sum(dout * O), O = attention(q, k, v).
    Query i and key j sit at positions i and j (upper-left causal).
    """
    lib = lib or load()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(dout)
    lead = q.shape[:-2]
    if k.shape[:-2] != lead or v.shape[:-2] != lead or g.shape[:-2] != lead:
        raise ValueError("leading axes differ")
    tq, d = q.shape[-2:]
    tk, dv = v.shape[-2:]
    if k.shape[-1] != d or k.shape[-2] != tk or g.shape[-2:] != (tq, dv):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bh = int(np.prod(lead)) if lead else 1
    dq, dk, dvv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    rc = lib.oracle_attention_grad(bh, tq, tk, d, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                   int(bool(causal)), float(scale), _ptr(dq), _ptr(dk),
                                   _ptr(dvv))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_grad failed ({rc})")
    return dq, dk, dvv


def grad_query_rows(q_rows, dout_rows, q_pos, k, v, causal=False, scale=None, lib=None):
    """dQ of selected query rows of ONE head, with each row's lse and D.

    q_rows [R, d], dout_rows [R, dv], positions q_pos [R]; k [Tk, d],
    v [Tk, dv] -> (dq [R, d], lse [R], delta [R]).
    """
    lib = lib or load()
    q_rows, g, k, v = _f64(q_rows), _f64(dout_rows), _f64(k), _f64(v)
    pos = np.ascontiguousarray(np.asarray(q_pos, dtype=np.int64))
    r, d = q_rows.shape
    tk, dv = v.shape
    if pos.shape != (r,) or k.shape != (tk, d) or g.shape != (r, dv):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, lse, delta = np.zeros((r, d)), np.zeros(r), np.zeros(r)
    rc = lib.oracle_grad_query_rows(tk, d, dv, _ptr(k), _ptr(v), r, _ptr(q_rows), _ptr(g),
                                    _ptr(pos), int(bool(causal)), float(scale), _ptr(dq),
                                    _ptr(lse), _ptr(delta))
    if rc != 0:
        raise RuntimeError(f"oracle_grad_query_rows failed ({rc})")
    return dq, lse, delta


def grad_key_rows(k_rows, v_rows, k_pos, q, dout, lse, delta, causal=False, scale=None,
                  lib=None):
    """dK, dV of selected key rows of ONE head.

    k_rows [R, d], v_rows [R, dv], positions k_pos [R]; all queries of the
    head q [Tq, d], dout [Tq, dv] with their lse [Tq] and delta [Tq] (from
    ``grad_query_rows`` over every query) -> (dk [R, d], dv [R, dv]).
    """
    lib = lib or load()
    k_rows, v_rows, q, g = _f64(k_rows), _f64(v_rows), _f64(q), _f64(dout)
    lse, delta = _f64(lse), _f64(delta)
    pos = np.ascontiguousarray(np.asarray(k_pos, dtype=np.int64))
    r, d = k_rows.shape
    tq, dv = g.shape
    if pos.shape != (r,) or v_rows.shape != (r, dv) or q.shape != (tq, d) or \
            lse.shape != (tq,) or delta.shape != (tq,):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dk, dvv = np.zeros((r, d)), np.zeros((r, dv))
    rc = lib.oracle_grad_key_rows(tq, d, dv, _ptr(q), _ptr(g), _ptr(lse), _ptr(delta), r,
                                  _ptr(k_rows), _ptr(v_rows), _ptr(pos), int(bool(causal)),
                                  float(scale), _ptr(dk), _ptr(dvv))
    if rc != 0:
        raise RuntimeError(f"oracle_grad_key_rows failed ({rc})")
    return dk, dvv


def dropout_threshold(p):
    """Byte threshold t = floor((1 - p) * 256 + 1/2) of the keep rule (keep
    iff the element's random byte < t); dropout probability p must be in
    [0, 1) and leave t >= 1."""
    if not (0.0 <= float(p) < 1.0):
        raise ValueError("dropout probability must be in [0, 1)")
    t = int(math.floor((1.0 - float(p)) * 256.0 + 0.5))
    if t < 1:
        raise ValueError("dropout probability leaves no weight kept (t = 0)")
    return t


def philox4x32_10(ctr, key, lib=None):
    """The four 32-bit words of Philox4x32-10 for counter ctr[4], key key[2]."""
    lib = lib or load()
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(c.ctypes.data_as(ctypes.c_void_p), k.ctypes.data_as(ctypes.c_void_p),
                             out.ctypes.data_as(ctypes.c_void_p))
    return out


def dropout_mask(bh, nq, nk, seed, offset, p, lib=None):
    """Keep mask [nq, nk] (uint8 0/1) of head ``bh`` (small shapes)."""
    lib = lib or load()
    mask = np.zeros((nq, nk), dtype=np.uint8)
    rc = lib.oracle_dropout_mask(int(bh), int(nq), int(nk), int(seed), int(offset),
                                 dropout_threshold(p), _ptr(mask))
    if rc != 0:
        raise RuntimeError(f"oracle_dropout_mask failed ({rc})")
    return mask


def attention_dropout(q, k, v, bh, seed, offset, p, causal=False, scale=None, lib=None,
                      q_offset=0):
    """O, LSE of ONE head (q [Tq, d], k [Tk, d], v [Tk, dv]; head index ``bh``
    in the batch*head numbering the mask is drawn with) with dropout
    probability p on the attention weights.  Query row i sits at position
    i + q_offset (causal: keys j <= i + q_offset); the mask is indexed by
    the row i and the key j whatever the offset."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    tq, d = q.shape
    tk, dv = v.shape
    if k.shape != (tk, d):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o, lse = np.zeros((tq, dv)), np.zeros(tq)
    rc = lib.oracle_attention_dropout(int(bh), tq, tk, d, dv, _ptr(q), _ptr(k), _ptr(v),
                                      int(bool(causal)), int(q_offset), float(scale), int(seed),
                                      int(offset), dropout_threshold(p), _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_dropout failed ({rc})")
    return o, lse


def attention_dropout_grad(q, k, v, dout, bh, seed, offset, p, causal=False, scale=None,
                           lib=None, q_offset=0):
    """dQ, dK, dV of sum(dout * O) for O = attention_dropout(...) of ONE head
    (query row i at position i + q_offset)."""
    lib = lib or load()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(dout)
    tq, d = q.shape
    tk, dv = v.shape
    if k.shape != (tk, d) or g.shape != (tq, dv):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dvv = np.zeros((tq, d)), np.zeros((tk, d)), np.zeros((tk, dv))
    rc = lib.oracle_attention_dropout_grad(int(bh), tq, tk, d, dv, _ptr(q), _ptr(k), _ptr(v),
                                           _ptr(g), int(bool(causal)), int(q_offset), float(scale),
                                           int(seed), int(offset), dropout_threshold(p), _ptr(dq),
                                           _ptr(dk), _ptr(dvv))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_dropout_grad failed ({rc})")
    return dq, dk, dvv
