"""Float64 CPU oracle for exact attention.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never import, link or call it, and it imports nothing from them.

* ``attention`` / ``attention_rows`` — the plain definition (scores, row max,
  exp-sum, V blend, logsumexp) in C, ``attn_oracle.c``.
* ``online_model`` — the block-wise online recurrence in numpy, the second
  derivation the C code is pinned against.

``build()`` compiles ``attn_oracle.c`` with gcc (OpenMP over rows) into
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
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None


def compile_oracle(src=_SRC, out=_LIB_PATH, extra_flags=()):
    """Compile an oracle source file into a shared library; returns the path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99", *extra_flags,
           src, "-o", out + ".tmp", "-lm"]
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
    return lib


def load(path=None):
    """The compiled oracle (building it first when it is missing)."""
    global _lib
    if path is not None:
        return _bind(path)
    if _lib is None:
        if not os.path.exists(_LIB_PATH) or (
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
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
