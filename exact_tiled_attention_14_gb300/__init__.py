"""Exact tiled attention for GB300 (sm_103a): Python binding.

This module only marshals arguments to the C ABI in ``include/fa.h``
(every name in ``EXPORTS``: the forward entry points ``fa_fwd``,
``fa_fwd_ws``, ``fa_fwd_static``, ``fa_fwd_kv``, ``fa_fwd_varlen`` and their
``_dropout`` forms; the backward ``fa_bwd``, ``fa_bwd_kv``, ``fa_bwd_varlen``,
their ``_dropout`` forms, ``fa_bwd_onepass`` and ``fa_bwd_onepass_dropout``;
``fa_decode``; the workspace sizes, status and settings), under the same
names.  Every step of
the attention computation runs in the CUDA kernels of ``_build/libfa.so``;
there is no CPU or PyTorch fallback.  When the library has not been built,
every call raises.

``attention_forward`` is the convenience call a user makes: it allocates O
and LSE (and, when asked, the balancing workspace) with PyTorch — device
memory is PyTorch's job here — and calls ``fa_fwd`` or ``fa_fwd_ws`` on the
current CUDA stream.  ``attention_backward`` does the same for ``fa_bwd``
(dQ, dK, dV and the D scratch), ``attention_decode`` for ``fa_decode``,
``attention_forward_kv`` for ``fa_fwd_kv``, ``attention_forward_varlen`` for
``fa_fwd_varlen``, ``attention_backward_onepass`` for ``fa_bwd_onepass``
(and ``fa_bwd_onepass_dropout``).  ``flash_attention``, ``flash_attention_kv`` and
``flash_attention_varlen`` wrap the forward and backward entry points in
torch.autograd functions.
"""
import ctypes
import math
import os

from .build import LIB_PATH, build  # noqa: F401

FA_BF16 = 0
FA_FP16 = 1

FA_OK = 0
FA_ERR_NULLPTR = 1
FA_ERR_SHAPE = 2
FA_ERR_UNSUPPORTED_D = 3
FA_ERR_DTYPE = 4
FA_ERR_ALIGN = 5
FA_ERR_SCALE = 6
FA_ERR_DEVICE = 7
FA_ERR_TENSORMAP = 8
FA_ERR_LAUNCH = 9
FA_ERR_TIMEOUT = 10
FA_ERR_CUDA = 11
FA_ERR_WORKSPACE = 12
FA_ERR_DROPOUT = 13

# Functions the C ABI exports (checked against include/fa.h by the tests).
EXPORTS = ("fa_fwd", "fa_fwd_kv", "fa_fwd_varlen", "fa_fwd_dropout", "fa_bwd_dropout", "fa_bwd_kv", "fa_bwd_varlen",
           "fa_fwd_kv_dropout", "fa_fwd_varlen_dropout", "fa_bwd_kv_dropout",
           "fa_bwd_varlen_dropout",
           "fa_fwd_ws", "fa_fwd_workspace_size", "fa_fwd_static", "fa_bwd",
           "fa_bwd_onepass", "fa_bwd_onepass_workspace_size", "fa_bwd_onepass_dropout",
           "fa_decode", "fa_decode_workspace_size", "fa_strerror", "fa_status",
           "fa_set_watchdog_ns", "fa_set_unit_group", "fa_watchdog_selftest", "fa_work_tiles",
           "fa_version")

_lib = None


class FaError(RuntimeError):
    """A non-zero return code of the C ABI."""

    def __init__(self, code, where="fa_fwd"):
        self.code = int(code)
        super().__init__(f"{where}: {fa_strerror(self.code)} (code {self.code})")


def load_library(path=None):
    """Load ``libfa.so`` (raises if it has not been built)."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library not built: {p} is missing "
            "(run exact_tiled_attention_14_gb300.build.build())")
    lib = ctypes.CDLL(p)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_kv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, f, i, vp]
    lib.fa_fwd_kv.restype = i
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_fwd_ws.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_ws.restype = i
    lib.fa_fwd_workspace_size.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_fwd_workspace_size.restype = i
    lib.fa_fwd_static.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_static.restype = i
    lib.fa_bwd.argtypes = [vp] * 10 + [i, i, i, i, i, f, i, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_onepass.argtypes = [vp] * 10 + [i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
    lib.fa_bwd_onepass.restype = i
    lib.fa_bwd_onepass_workspace_size.argtypes = [i] * 4 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_bwd_onepass_workspace_size.restype = i
    u64, u32 = ctypes.c_ulonglong, ctypes.c_uint
    lib.fa_bwd_onepass_dropout.argtypes = ([vp] * 10 + [i, i, i, i, i, f, f, u64, u32, i, vp,
                                                         ctypes.c_size_t, vp])
    lib.fa_bwd_onepass_dropout.restype = i
    lib.fa_fwd_dropout.argtypes = [vp] * 5 + [i, i, i, i, i, f, f, u64, u32, i, vp]
    lib.fa_fwd_dropout.restype = i
    lib.fa_bwd_dropout.argtypes = [vp] * 10 + [i, i, i, i, i, f, f, u64, u32, i, vp]
    lib.fa_bwd_dropout.restype = i
    lib.fa_fwd_kv_dropout.argtypes = [vp] * 5 + [i] * 7 + [vp, f, f, u64, u32, i, vp]
    lib.fa_fwd_kv_dropout.restype = i
    lib.fa_fwd_varlen_dropout.argtypes = [vp] * 7 + [i] * 8 + [f, f, u64, u32, i, vp]
    lib.fa_fwd_varlen_dropout.restype = i
    lib.fa_bwd_kv_dropout.argtypes = [vp] * 10 + [i] * 7 + [vp, f, f, u64, u32, i, vp]
    lib.fa_bwd_kv_dropout.restype = i
    lib.fa_bwd_varlen_dropout.argtypes = [vp] * 12 + [i] * 9 + [f, f, u64, u32, i, vp]
    lib.fa_bwd_varlen_dropout.restype = i
    lib.fa_bwd_kv.argtypes = [vp] * 10 + [i, i, i, i, i, i, i, vp, f, i, vp]
    lib.fa_bwd_kv.restype = i
    lib.fa_bwd_varlen.argtypes = [vp] * 12 + [i] * 9 + [f, i, vp]
    lib.fa_bwd_varlen.restype = i
    lib.fa_decode.argtypes = [vp] * 5 + [i] * 6 + [f, i, vp, ctypes.c_size_t, vp]
    lib.fa_decode.restype = i
    lib.fa_decode_workspace_size.argtypes = [i] * 5 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_decode_workspace_size.restype = i
    lib.fa_strerror.argtypes = [i]
    lib.fa_strerror.restype = ctypes.c_char_p
    lib.fa_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.fa_status.restype = i
    lib.fa_set_watchdog_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_set_watchdog_ns.restype = None
    lib.fa_set_unit_group.argtypes = [ctypes.c_int]
    lib.fa_set_unit_group.restype = ctypes.c_int
    lib.fa_watchdog_selftest.argtypes = [ctypes.c_ulonglong, vp]
    lib.fa_watchdog_selftest.restype = i
    lib.fa_work_tiles.argtypes = [i, i, ctypes.POINTER(ctypes.c_longlong)]
    lib.fa_work_tiles.restype = i
    lib.fa_version.argtypes = []
    lib.fa_version.restype = i
    if path is None:
        _lib = lib
    return lib


def _addr(x):
    """Device address of a tensor, or an int / None passed through."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, stream=None):
    """Raw C call; tensors or integer addresses; returns the C return code."""
    lib = load_library()
    return lib.fa_fwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                      int(N), int(d), int(bool(causal)), float(scale), int(dtype),
                      _stream(stream))


def fa_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, dv, causal, seqlens_k, scale, dtype,
              stream=None):
    """Raw C call: Nq queries of width d against Nk keys, values of width dv
    (seqlens_k: per-batch key counts or None; causal 0 none, 1 upper-left,
    2 bottom-right); returns the code."""
    lib = load_library()
    return lib.fa_fwd_kv(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                         int(Nq), int(Nk), int(d), int(dv), int(causal), _addr(seqlens_k),
                         float(scale), int(dtype), _stream(stream))


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, total_q,
                  total_k, d, dv, causal, scale, dtype, stream=None):
    """Raw C call: packed sequences (token-major q, k, v, o; lse [H, total_q];
    cu_seqlens_* int32 offsets, B + 1 each); returns the code."""
    lib = load_library()
    return lib.fa_fwd_varlen(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse),
                             _addr(cu_seqlens_q), _addr(cu_seqlens_k), int(B), int(H),
                             int(max_seqlen_q), int(total_q), int(total_k), int(d), int(dv),
                             int(causal), float(scale), int(dtype), _stream(stream))


def fa_fwd_ws(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, workspace, workspace_bytes,
              stream=None):
    """Raw C call with a balancing workspace; returns the C return code."""
    lib = load_library()
    return lib.fa_fwd_ws(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                         int(N), int(d), int(bool(causal)), float(scale), int(dtype),
                         _addr(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_static(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, stream=None):
    """Raw C call of the entry point that allocates nothing (library-held scratch)."""
    lib = load_library()
    return lib.fa_fwd_static(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                             int(N), int(d), int(bool(causal)), float(scale), int(dtype),
                             _stream(stream))


def fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, causal, scale, dropout_p, seed, offset, dtype,
                   stream=None):
    """Raw C call of the forward pass with dropout; returns the code."""
    lib = load_library()
    return lib.fa_fwd_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                              int(N), int(d), int(bool(causal)), float(scale), float(dropout_p),
                              int(seed), int(offset), int(dtype), _stream(stream))


def fa_bwd_dropout(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, d, causal, scale,
                   dropout_p, seed, offset, dtype, stream=None):
    """Raw C call of the backward pass with dropout; returns the code."""
    lib = load_library()
    return lib.fa_bwd_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dout),
                              _addr(dq), _addr(dk), _addr(dv), _addr(delta), int(B), int(H),
                              int(N), int(d), int(bool(causal)), float(scale), float(dropout_p),
                              int(seed), int(offset), int(dtype), _stream(stream))


def fa_fwd_kv_dropout(q, k, v, o, lse, B, H, Nq, Nk, d, dv, causal, seqlens_k, scale, dropout_p,
                      seed, offset, dtype, stream=None):
    """Raw C call of fa_fwd_kv with dropout on the attention weights; returns the code."""
    lib = load_library()
    return lib.fa_fwd_kv_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B),
                                 int(H), int(Nq), int(Nk), int(d), int(dv), int(causal),
                                 _addr(seqlens_k), float(scale), float(dropout_p), int(seed),
                                 int(offset), int(dtype), _stream(stream))


def fa_fwd_varlen_dropout(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q,
                          total_q, total_k, d, dv, causal, scale, dropout_p, seed, offset, dtype,
                          stream=None):
    """Raw C call of fa_fwd_varlen with dropout on the attention weights; returns the code."""
    lib = load_library()
    return lib.fa_fwd_varlen_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse),
                                     _addr(cu_seqlens_q), _addr(cu_seqlens_k), int(B), int(H),
                                     int(max_seqlen_q), int(total_q), int(total_k), int(d),
                                     int(dv), int(causal), float(scale), float(dropout_p),
                                     int(seed), int(offset), int(dtype), _stream(stream))


def fa_bwd_kv_dropout(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, d, dv_width,
                      causal, seqlens_k, scale, dropout_p, seed, offset, dtype, stream=None):
    """Raw C call of the backward pass of fa_fwd_kv_dropout; returns the code."""
    lib = load_library()
    return lib.fa_bwd_kv_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dout),
                                 _addr(dq), _addr(dk), _addr(dv), _addr(delta), int(B), int(H),
                                 int(Nq), int(Nk), int(d), int(dv_width), int(causal),
                                 _addr(seqlens_k), float(scale), float(dropout_p), int(seed),
                                 int(offset), int(dtype), _stream(stream))


def fa_bwd_varlen_dropout(q, k, v, o, lse, dout, dq, dk, dv, delta, cu_seqlens_q, cu_seqlens_k, B,
                          H, max_seqlen_q, max_seqlen_k, total_q, total_k, d, dv_width, causal,
                          scale, dropout_p, seed, offset, dtype, stream=None):
    """Raw C call of the backward pass of fa_fwd_varlen_dropout; returns the code."""
    lib = load_library()
    return lib.fa_bwd_varlen_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse),
                                     _addr(dout), _addr(dq), _addr(dk), _addr(dv), _addr(delta),
                                     _addr(cu_seqlens_q), _addr(cu_seqlens_k), int(B), int(H),
                                     int(max_seqlen_q), int(max_seqlen_k), int(total_q),
                                     int(total_k), int(d), int(dv_width), int(causal),
                                     float(scale), float(dropout_p), int(seed), int(offset),
                                     int(dtype), _stream(stream))


def fa_bwd_kv(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, d, dv_width, causal,
              seqlens_k, scale, dtype, stream=None):
    """Raw C call of the backward pass of fa_fwd_kv (query/key width d, value
    width dv_width); returns the code."""
    lib = load_library()
    return lib.fa_bwd_kv(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dout),
                         _addr(dq), _addr(dk), _addr(dv), _addr(delta), int(B), int(H), int(Nq),
                         int(Nk), int(d), int(dv_width), int(causal), _addr(seqlens_k),
                         float(scale), int(dtype), _stream(stream))


def fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, delta, cu_seqlens_q, cu_seqlens_k, B, H,
                  max_seqlen_q, max_seqlen_k, total_q, total_k, d, dv_width, causal, scale, dtype,
                  stream=None):
    """Raw C call of the backward pass of fa_fwd_varlen (query/key width d,
    value width dv_width); returns the code."""
    lib = load_library()
    return lib.fa_bwd_varlen(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dout),
                             _addr(dq), _addr(dk), _addr(dv), _addr(delta), _addr(cu_seqlens_q),
                             _addr(cu_seqlens_k), int(B), int(H), int(max_seqlen_q),
                             int(max_seqlen_k), int(total_q), int(total_k), int(d), int(dv_width),
                             int(causal), float(scale), int(dtype), _stream(stream))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, d, causal, scale, dtype,
           stream=None):
    """Raw C call of the backward pass; tensors or integer addresses; returns the code."""
    lib = load_library()
    return lib.fa_bwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dout), _addr(dq),
                      _addr(dk), _addr(dv), _addr(delta), int(B), int(H), int(N), int(d),
                      int(bool(causal)), float(scale), int(dtype), _stream(stream))


def fa_bwd_onepass(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, d, causal, scale, dtype,
                   workspace, workspace_bytes, stream=None):
    """Raw C call of the one-pass backward; tensors or integer addresses; returns the code."""
    lib = load_library()
    return lib.fa_bwd_onepass(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dout),
                              _addr(dq), _addr(dk), _addr(dv), _addr(delta), int(B), int(H),
                              int(N), int(d), int(bool(causal)), float(scale), int(dtype),
                              _addr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_onepass_dropout(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, d, causal, scale,
                           dropout_p, seed, offset, dtype, workspace, workspace_bytes,
                           stream=None):
    """Raw C call of the one-pass backward with dropout; returns the code."""
    lib = load_library()
    return lib.fa_bwd_onepass_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse),
                                      _addr(dout), _addr(dq), _addr(dk), _addr(dv), _addr(delta),
                                      int(B), int(H), int(N), int(d), int(bool(causal)),
                                      float(scale), float(dropout_p), int(seed), int(offset),
                                      int(dtype), _addr(workspace), int(workspace_bytes),
                                      _stream(stream))


def fa_bwd_onepass_workspace_size(B, H, N, d):
    """Bytes of the fp32 dQ sum fa_bwd_onepass needs for this shape."""
    out = ctypes.c_size_t(0)
    code = load_library().fa_bwd_onepass_workspace_size(int(B), int(H), int(N), int(d),
                                                        ctypes.byref(out))
    if code:
        raise FaError(code, "fa_bwd_onepass_workspace_size")
    return out.value


def fa_decode(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
              workspace_bytes, stream=None):
    """Raw C call of split-KV decoding; tensors or integer addresses; returns the code."""
    lib = load_library()
    return lib.fa_decode(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                         int(Nq), int(Nk), int(d), int(bool(causal)), float(scale), int(dtype),
                         _addr(workspace), int(workspace_bytes), _stream(stream))


def fa_decode_workspace_size(B, H, Nq, Nk, d):
    """Workspace bytes fa_decode needs for this shape on the current device."""
    out = ctypes.c_size_t(0)
    code = load_library().fa_decode_workspace_size(int(B), int(H), int(Nq), int(Nk), int(d),
                                                   ctypes.byref(out))
    if code:
        raise FaError(code, "fa_decode_workspace_size")
    return out.value


def fa_fwd_workspace_size(B, H, N, d, causal):
    """Workspace bytes fa_fwd_ws needs for this shape on the current device."""
    out = ctypes.c_size_t(0)
    code = load_library().fa_fwd_workspace_size(int(B), int(H), int(N), int(d),
                                                int(bool(causal)), ctypes.byref(out))
    if code:
        raise FaError(code, "fa_fwd_workspace_size")
    return out.value


def make_workspace(B, H, N, d, causal, device=None):
    """A device workspace (uint8 tensor) sized for fa_fwd_ws, or None if none is needed."""
    import torch
    n = fa_fwd_workspace_size(B, H, N, d, causal)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def fa_strerror(code):
    return load_library().fa_strerror(int(code)).decode()


def fa_status(stream=None):
    """(code, raw status word) after synchronising ``stream``."""
    detail = ctypes.c_uint(0)
    code = load_library().fa_status(_stream(stream), ctypes.byref(detail))
    return code, detail.value


def fa_set_watchdog_ns(ns):
    load_library().fa_set_watchdog_ns(int(ns))


def fa_set_unit_group(heads):
    """Unit-order override for the forward kernels (0 = choose per call);
    returns the C return code."""
    return load_library().fa_set_unit_group(int(heads))


def fa_watchdog_selftest(budget_ns, stream=None):
    """Launch the failure-detection self-test (a wait that must run out)."""
    return load_library().fa_watchdog_selftest(int(budget_ns), _stream(stream))


def fa_work_tiles(N, causal):
    out = ctypes.c_longlong(0)
    code = load_library().fa_work_tiles(int(N), int(bool(causal)), ctypes.byref(out))
    if code:
        raise FaError(code, "fa_work_tiles")
    return out.value


def fa_version():
    return load_library().fa_version()


def dtype_code(torch_dtype):
    import torch
    if torch_dtype == torch.bfloat16:
        return FA_BF16
    if torch_dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"unsupported dtype {torch_dtype}; use bfloat16 or float16")


def attention_forward(q, k, v, causal=False, scale=None, out=None, lse=None, stream=None,
                      workspace=None):
    """O, LSE = exact attention of CUDA tensors q, k, v [B, H, N, d].

    O has the input dtype; LSE is float32 [B, H, N] (natural log).  ``scale``
    defaults to 1/sqrt(d).  Runs on ``stream`` (default: current stream).
    ``workspace``: None runs ``fa_fwd``; a uint8 CUDA tensor (see
    ``make_workspace``) or ``"auto"`` (allocate one) runs ``fa_fwd_ws``, which
    balances the last round of work across the SMs.
    """
    import torch
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError(f"dtypes differ: {q.dtype}, {k.dtype}, {v.dtype}")
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must all be [B, H, N, d] of one shape")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    code = dtype_code(q.dtype)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if workspace is None:
        rc = fa_fwd(q, k, v, out, lse, B, H, N, d, causal, scale, code, stream)
    else:
        if isinstance(workspace, str):
            if workspace != "auto":
                raise ValueError("workspace must be None, 'auto' or a CUDA tensor")
            workspace = make_workspace(B, H, N, d, causal, device=q.device)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        rc = fa_fwd_ws(q, k, v, out, lse, B, H, N, d, causal, scale, code, workspace, ws_bytes,
                       stream)
    if rc != FA_OK:
        raise FaError(rc)
    return out, lse


CAUSAL_MODES = {None: 0, False: 0, "upper_left": 1, "bottom_right": 2}


def attention_forward_kv(q, k, v, causal=None, seqlens_k=None, scale=None, out=None, lse=None,
                         stream=None, dropout_p=0.0, seed=0, offset=0):
    """O [B, H, Nq, dv], LSE of queries q [B, H, Nq, d] against keys
    k [B, H, Nk, d] and values v [B, H, Nk, dv] (CUDA, contiguous, one 16-bit
    dtype; d and dv each 64 or 128).

    ``causal``: None (no mask), "upper_left" (query i at position i) or
    "bottom_right" (query i at position len_b - Nq + i).  ``seqlens_k``: None
    or an int32 CUDA tensor [B] of key counts per batch (the rest of the Nk
    keys is padding).  A query that sees no key gets O = 0 and LSE = -inf.
    Calls ``fa_fwd_kv`` on ``stream`` (default: current stream), or
    ``fa_fwd_kv_dropout`` when ``dropout_p`` > 0 (mask from seed, offset).
    """
    import torch
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError(f"dtypes differ: {q.dtype}, {k.dtype}, {v.dtype}")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4 or k.shape[:3] != v.shape[:3]:
        raise ValueError("q must be [B, H, Nq, d], k [B, H, Nk, d] and v [B, H, Nk, dv]")
    if q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q and k differ in batch, heads or head width")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if causal not in CAUSAL_MODES:
        raise ValueError("causal must be None, 'upper_left' or 'bottom_right'")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dv = v.shape[3]
    if seqlens_k is not None:
        if seqlens_k.dtype != torch.int32 or seqlens_k.shape != (B,) or not seqlens_k.is_cuda:
            raise ValueError("seqlens_k must be an int32 CUDA tensor of shape [B]")
        seqlens_k = seqlens_k.contiguous()
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, Nq, dv), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if dropout_p > 0:
        rc = fa_fwd_kv_dropout(q, k, v, out, lse, B, H, Nq, Nk, d, dv, CAUSAL_MODES[causal],
                               seqlens_k, scale, dropout_p, seed, offset, dtype_code(q.dtype),
                               stream)
    else:
        rc = fa_fwd_kv(q, k, v, out, lse, B, H, Nq, Nk, d, dv, CAUSAL_MODES[causal], seqlens_k,
                       scale, dtype_code(q.dtype), stream)
    if rc != FA_OK:
        raise FaError(rc)
    return out, lse


def attention_forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, causal=None,
                             scale=None, out=None, lse=None, stream=None, dropout_p=0.0, seed=0,
                             offset=0):
    """O [total_q, H, dv], LSE [H, total_q] of a packed batch: q [total_q, H, d],
    k [total_k, H, d], v [total_k, H, dv] (CUDA, contiguous, one 16-bit dtype);
    cu_seqlens_q / cu_seqlens_k int32 CUDA tensors [B + 1] of token offsets;
    ``max_seqlen_q`` (a host int) bounds every sequence's query count.

    ``causal``: None, "upper_left" or "bottom_right" (per sequence).  A
    query that sees no key gets O = 0 and LSE = -inf.  Calls ``fa_fwd_varlen``
    on ``stream`` (default: current stream).
    """
    import torch
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError(f"dtypes differ: {q.dtype}, {k.dtype}, {v.dtype}")
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or k.shape[:2] != v.shape[:2]:
        raise ValueError("q must be [total_q, H, d], k [total_k, H, d] and v [total_k, H, dv]")
    if q.shape[1] != k.shape[1] or q.shape[2] != k.shape[2]:
        raise ValueError("q and k differ in heads or head width")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if causal not in CAUSAL_MODES:
        raise ValueError("causal must be None, 'upper_left' or 'bottom_right'")
    for name, cu in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if cu.dtype != torch.int32 or cu.dim() != 1 or not cu.is_cuda or not cu.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor [B + 1]")
    if cu_seqlens_q.shape != cu_seqlens_k.shape or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 entries")
    total_q, H, d = q.shape
    total_k, dv = k.shape[0], v.shape[2]
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((total_q, H, dv), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if dropout_p > 0:
        rc = fa_fwd_varlen_dropout(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, B, H,
                                   int(max_seqlen_q), total_q, total_k, d, dv,
                                   CAUSAL_MODES[causal], scale, dropout_p, seed, offset,
                                   dtype_code(q.dtype), stream)
    else:
        rc = fa_fwd_varlen(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, B, H, int(max_seqlen_q),
                           total_q, total_k, d, dv, CAUSAL_MODES[causal], scale,
                           dtype_code(q.dtype), stream)
    if rc != FA_OK:
        raise FaError(rc)
    return out, lse


def attention_backward(q, k, v, o, lse, dout, causal=False, scale=None, stream=None):
    """dQ, dK, dV of sum(dout * O) for O, LSE = attention_forward(q, k, v).

    All tensors are CUDA [B, H, N, d] of one 16-bit dtype except lse (float32
    [B, H, N]).  Allocates dq, dk, dv and the float32 D scratch with PyTorch
    and calls ``fa_bwd`` on ``stream`` (default: current stream).
    """
    import torch
    ts = (q, k, v, o, dout)
    if any(t.dtype != q.dtype for t in ts):
        raise TypeError("q, k, v, o, dout must share one dtype")
    if q.dim() != 4 or any(t.shape != q.shape for t in ts):
        raise ValueError("q, k, v, o, dout must all be [B, H, N, d] of one shape")
    if lse.dtype != torch.float32 or lse.shape != q.shape[:3]:
        raise ValueError("lse must be float32 [B, H, N]")
    if not all(t.is_cuda and t.is_contiguous() for t in ts + (lse,)):
        raise ValueError("all tensors must be contiguous CUDA tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    code = dtype_code(q.dtype)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    rc = fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, d, causal, scale, code, stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def attention_backward_onepass(q, k, v, o, lse, dout, causal=False, scale=None, workspace=None,
                               stream=None, dropout_p=0.0, seed=0, offset=0):
    """The gradients of ``attention_backward`` (or, with dropout_p > 0, of
    ``attention_backward_dropout``) through ``fa_bwd_onepass`` (or
    ``fa_bwd_onepass_dropout``): each (query tile, key tile) pair is visited
    once and dQ is summed in fp32 through ``workspace`` (a CUDA tensor of at
    least ``fa_bwd_onepass_workspace_size`` bytes; allocated here when
    None).  dQ may differ in its last bits from call to call; dK and dV do
    not."""
    import torch
    ts = (q, k, v, o, dout)
    if any(t.dtype != q.dtype for t in ts):
        raise TypeError("q, k, v, o, dout must share one dtype")
    if q.dim() != 4 or any(t.shape != q.shape for t in ts):
        raise ValueError("q, k, v, o, dout must all be [B, H, N, d] of one shape")
    if lse.dtype != torch.float32 or lse.shape != q.shape[:3]:
        raise ValueError("lse must be float32 [B, H, N]")
    if not all(t.is_cuda and t.is_contiguous() for t in ts + (lse,)):
        raise ValueError("all tensors must be contiguous CUDA tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    code = dtype_code(q.dtype)
    need = fa_bwd_onepass_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if dropout_p > 0:
        rc = fa_bwd_onepass_dropout(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, d, causal,
                                    scale, dropout_p, seed, offset, code, workspace, ws_bytes,
                                    stream)
    else:
        rc = fa_bwd_onepass(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, d, causal, scale,
                            code, workspace, ws_bytes, stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_onepass_dropout" if dropout_p > 0 else "fa_bwd_onepass")
    return dq, dk, dv


def attention_forward_dropout(q, k, v, dropout_p, seed, offset, causal=False, scale=None,
                              out=None, lse=None, stream=None):
    """O, LSE of ``attention_forward`` with dropout on the attention weights
    (``fa_fwd_dropout``): the same (dropout_p, seed, offset) given to
    ``attention_backward_dropout`` regenerate the mask."""
    import torch
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError(f"dtypes differ: {q.dtype}, {k.dtype}, {v.dtype}")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must be [B, H, N, d] of one shape")
    if not all(t.is_cuda and t.is_contiguous() for t in (q, k, v)):
        raise ValueError("q, k, v must be contiguous CUDA tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    rc = fa_fwd_dropout(q, k, v, out, lse, B, H, N, d, causal, scale, dropout_p, seed, offset,
                        dtype_code(q.dtype), stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_dropout")
    return out, lse


def attention_backward_dropout(q, k, v, o, lse, dout, dropout_p, seed, offset, causal=False,
                               scale=None, stream=None):
    """dQ, dK, dV for O, LSE = attention_forward_dropout(q, k, v, dropout_p,
    seed, offset) (``fa_bwd_dropout``; the mask is regenerated)."""
    import torch
    ts = (q, k, v, o, dout)
    if any(t.dtype != q.dtype for t in ts):
        raise TypeError("q, k, v, o, dout must share one dtype")
    if q.dim() != 4 or any(t.shape != q.shape for t in ts):
        raise ValueError("q, k, v, o, dout must all be [B, H, N, d] of one shape")
    if lse.dtype != torch.float32 or lse.shape != q.shape[:3]:
        raise ValueError("lse must be float32 [B, H, N]")
    if not all(t.is_cuda and t.is_contiguous() for t in ts + (lse,)):
        raise ValueError("all tensors must be contiguous CUDA tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    rc = fa_bwd_dropout(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, d, causal, scale,
                        dropout_p, seed, offset, dtype_code(q.dtype), stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_dropout")
    return dq, dk, dv


def attention_backward_kv(q, k, v, o, lse, dout, causal=None, seqlens_k=None, scale=None,
                          stream=None, dropout_p=0.0, seed=0, offset=0):
    """dQ, dK, dV for O, LSE = attention_forward_kv(q, k, v, causal, seqlens_k)
    (``fa_bwd_kv``; q [B, H, Nq, d], k [B, H, Nk, d], v [B, H, Nk, dv],
    o, dout [B, H, Nq, dv]; d and dv each 64 or 128)."""
    import torch
    ts = (q, k, v, o, dout)
    if any(t.dtype != q.dtype for t in ts):
        raise TypeError("q, k, v, o, dout must share one dtype")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4 or k.shape[:3] != v.shape[:3] or \
            k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3] or \
            o.shape != q.shape[:3] + (v.shape[3],) or dout.shape != o.shape:
        raise ValueError("q must be [B, H, Nq, d], k [B, H, Nk, d], v [B, H, Nk, dv] and "
                         "o, dout [B, H, Nq, dv]")
    if lse.dtype != torch.float32 or lse.shape != q.shape[:3]:
        raise ValueError("lse must be float32 [B, H, Nq]")
    if not all(t.is_cuda and t.is_contiguous() for t in ts + (lse,)):
        raise ValueError("all tensors must be contiguous CUDA tensors")
    if causal not in CAUSAL_MODES:
        raise ValueError("causal must be None, 'upper_left' or 'bottom_right'")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if seqlens_k is not None:
        if seqlens_k.dtype != torch.int32 or seqlens_k.shape != (B,) or not seqlens_k.is_cuda:
            raise ValueError("seqlens_k must be an int32 CUDA tensor of shape [B]")
        seqlens_k = seqlens_k.contiguous()
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if dropout_p > 0:
        rc = fa_bwd_kv_dropout(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, d,
                               v.shape[3], CAUSAL_MODES[causal], seqlens_k, scale, dropout_p, seed,
                               offset, dtype_code(q.dtype), stream)
    else:
        rc = fa_bwd_kv(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, d, v.shape[3],
                       CAUSAL_MODES[causal], seqlens_k, scale, dtype_code(q.dtype), stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_kv")
    return dq, dk, dv


def attention_backward_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                              max_seqlen_k, causal=None, scale=None, stream=None, dropout_p=0.0,
                              seed=0, offset=0):
    """dQ, dK, dV for O, LSE = attention_forward_varlen(q, k, v, cu_seqlens_q,
    cu_seqlens_k, max_seqlen_q, causal) (``fa_bwd_varlen``; token-major
    [total, H, d] tensors, LSE [H, total_q]; max_seqlen_k a host int)."""
    import torch
    ts = (q, k, v, o, dout)
    if any(t.dtype != q.dtype for t in ts):
        raise TypeError("q, k, v, o, dout must share one dtype")
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3 or k.shape[:2] != v.shape[:2] or \
            k.shape[1:] != q.shape[1:] or o.shape != q.shape[:2] + (v.shape[2],) or \
            dout.shape != o.shape:
        raise ValueError("q must be [total_q, H, d], k [total_k, H, d], v [total_k, H, dv] and "
                         "o, dout [total_q, H, dv]")
    if lse.dtype != torch.float32 or lse.shape != (q.shape[1], q.shape[0]):
        raise ValueError("lse must be float32 [H, total_q]")
    if not all(t.is_cuda and t.is_contiguous() for t in ts + (lse,)):
        raise ValueError("all tensors must be contiguous CUDA tensors")
    if causal not in CAUSAL_MODES:
        raise ValueError("causal must be None, 'upper_left' or 'bottom_right'")
    for name, cu in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if cu.dtype != torch.int32 or cu.dim() != 1 or not cu.is_cuda or not cu.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor [B + 1]")
    if cu_seqlens_q.shape != cu_seqlens_k.shape or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 entries")
    total_q, H, d = q.shape
    total_k = k.shape[0]
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((total_q, H), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if dropout_p > 0:
        rc = fa_bwd_varlen_dropout(q, k, v, o, lse, dout, dq, dk, dv, delta, cu_seqlens_q,
                                   cu_seqlens_k, B, H, int(max_seqlen_q), int(max_seqlen_k),
                                   total_q, total_k, d, v.shape[2], CAUSAL_MODES[causal], scale,
                                   dropout_p, seed, offset, dtype_code(q.dtype), stream)
    else:
        rc = fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, delta, cu_seqlens_q, cu_seqlens_k,
                           B, H, int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, d,
                           v.shape[2], CAUSAL_MODES[causal], scale, dtype_code(q.dtype), stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_varlen")
    return dq, dk, dv


def attention_decode(q, k, v, causal=False, scale=None, out=None, lse=None, workspace=None,
                     stream=None):
    """O, LSE of a few queries q [B, H, Nq, d] (Nq <= 16) against a cache
    k, v [B, H, Nk, d] with the key axis split across the GPU (``fa_decode``).

    ``causal``: query i sits at position Nk - Nq + i.  ``workspace``: a uint8
    CUDA tensor of at least ``fa_decode_workspace_size`` bytes, or None to
    allocate one.
    """
    import torch
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError(f"dtypes differ: {q.dtype}, {k.dtype}, {v.dtype}")
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or q.shape[:2] != k.shape[:2] \
            or q.shape[3] != k.shape[3]:
        raise ValueError("q must be [B, H, Nq, d] and k, v [B, H, Nk, d]")
    if not all(t.is_cuda and t.is_contiguous() for t in (q, k, v)):
        raise ValueError("q, k, v must be contiguous CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    code = dtype_code(q.dtype)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = fa_decode_workspace_size(B, H, Nq, Nk, d)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = fa_decode(q, k, v, out, lse, B, H, Nq, Nk, d, causal, scale, code, workspace, ws_bytes,
                   stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_decode")
    return out, lse


# ---------------------------------------------------------------- autograd
# torch.autograd wrappers: the forward entry point in forward(), the matching
# backward entry point in backward(), so a PyTorch training step can call
# the library directly.  They only route tensors to the C ABI; what is saved
# for backward is what the pages say a backward pass keeps (Q, K, V, O and
# the row statistics LSE, plus the dropout generator's seed and offset).

def _autograd():
    import torch

    class _FlashAttention(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, causal, scale, dropout_p, seed, offset):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            if dropout_p > 0:
                o, lse = attention_forward_dropout(q, k, v, dropout_p, seed, offset, causal=causal,
                                                   scale=scale)
            else:
                o, lse = attention_forward(q, k, v, causal=causal, scale=scale)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.args = (causal, scale, dropout_p, seed, offset)
            ctx.mark_non_differentiable(lse)
            return o, lse

        @staticmethod
        def backward(ctx, do, _dlse):
            q, k, v, o, lse = ctx.saved_tensors
            causal, scale, dropout_p, seed, offset = ctx.args
            do = do.contiguous()
            if dropout_p > 0:
                g = attention_backward_dropout(q, k, v, o, lse, do, dropout_p, seed, offset,
                                               causal=causal, scale=scale)
            else:
                g = attention_backward(q, k, v, o, lse, do, causal=causal, scale=scale)
            return g[0], g[1], g[2], None, None, None, None, None

    class _FlashAttentionKv(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, causal, seqlens_k, scale, dropout_p, seed, offset):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            o, lse = attention_forward_kv(q, k, v, causal=causal, seqlens_k=seqlens_k, scale=scale,
                                          dropout_p=dropout_p, seed=seed, offset=offset)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.args = (causal, seqlens_k, scale, dropout_p, seed, offset)
            ctx.mark_non_differentiable(lse)
            return o, lse

        @staticmethod
        def backward(ctx, do, _dlse):
            q, k, v, o, lse = ctx.saved_tensors
            causal, seqlens_k, scale, dropout_p, seed, offset = ctx.args
            g = attention_backward_kv(q, k, v, o, lse, do.contiguous(), causal=causal,
                                      seqlens_k=seqlens_k, scale=scale, dropout_p=dropout_p,
                                      seed=seed, offset=offset)
            return g[0], g[1], g[2], None, None, None, None, None, None

    class _FlashAttentionVarlen(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, cu_q, cu_k, max_q, max_k, causal, scale, dropout_p, seed,
                    offset):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            o, lse = attention_forward_varlen(q, k, v, cu_q, cu_k, max_q, causal=causal,
                                              scale=scale, dropout_p=dropout_p, seed=seed,
                                              offset=offset)
            ctx.save_for_backward(q, k, v, o, lse, cu_q, cu_k)
            ctx.args = (max_q, max_k, causal, scale, dropout_p, seed, offset)
            ctx.mark_non_differentiable(lse)
            return o, lse

        @staticmethod
        def backward(ctx, do, _dlse):
            q, k, v, o, lse, cu_q, cu_k = ctx.saved_tensors
            max_q, max_k, causal, scale, dropout_p, seed, offset = ctx.args
            g = attention_backward_varlen(q, k, v, o, lse, do.contiguous(), cu_q, cu_k, max_q,
                                          max_k, causal=causal, scale=scale, dropout_p=dropout_p,
                                          seed=seed, offset=offset)
            return g[0], g[1], g[2], None, None, None, None, None, None, None, None, None

    return _FlashAttention, _FlashAttentionKv, _FlashAttentionVarlen


_AUTOGRAD = None


def _fns():
    global _AUTOGRAD
    if _AUTOGRAD is None:
        _AUTOGRAD = _autograd()
    return _AUTOGRAD


def flash_attention(q, k, v, causal=False, scale=None, dropout_p=0.0, seed=0, offset=0):
    """Differentiable O, LSE of exact attention over [B, H, N, d] (fa_fwd, or
    fa_fwd_dropout when dropout_p > 0; the backward through fa_bwd /
    fa_bwd_dropout with the same seed and offset)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _fns()[0].apply(q, k, v, bool(causal), float(scale), float(dropout_p), int(seed),
                           int(offset))


def flash_attention_kv(q, k, v, causal=None, seqlens_k=None, scale=None, dropout_p=0.0, seed=0,
                       offset=0):
    """Differentiable O, LSE of queries [B, H, Nq, d] against keys [B, H, Nk, d]
    and values [B, H, Nk, dv] (fa_fwd_kv / fa_bwd_kv, or their dropout forms
    when dropout_p > 0)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _fns()[1].apply(q, k, v, causal, seqlens_k, float(scale), float(dropout_p), int(seed),
                           int(offset))


def flash_attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                           causal=None, scale=None, dropout_p=0.0, seed=0, offset=0):
    """Differentiable O [total_q, H, dv], LSE [H, total_q] of a packed batch
    (fa_fwd_varlen / fa_bwd_varlen, or their dropout forms when dropout_p > 0)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _fns()[2].apply(q, k, v, cu_seqlens_q, cu_seqlens_k, int(max_seqlen_q),
                           int(max_seqlen_k), causal, float(scale), float(dropout_p), int(seed),
                           int(offset))
