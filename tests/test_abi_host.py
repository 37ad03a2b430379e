"""Host-side checks of the C ABI (no GPU needed).

The shared library must load and export every function ``include/fa.h``
declares; argument errors must come back as return codes before any device
work; and the causal tile schedule must match the counts the pages print.
No test here launches a kernel.
"""
import ctypes
import os
import re
import subprocess

import pytest

import exact_tiled_attention_14_gb300 as fa
from oracle_pins import read_golden  # noqa: F401  (golden helpers live there)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.LIB_PATH):
        fa.build()
    return fa.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_\w+)\s*\(", text)))


def test_header_lists_the_binding_names():
    assert header_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_header_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(fa_\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_library_has_no_oracle_or_torch_dependency():
    out = subprocess.run(["nm", "-D", fa.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    assert "oracle_" not in out
    ldd = subprocess.run(["ldd", fa.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in ldd and "liboracle" not in ldd


def test_strerror_covers_codes(lib):
    for code in range(0, fa.FA_ERR_DROPOUT + 1):
        s = fa.fa_strerror(code)
        assert s and s != "unknown error code"
    assert fa.fa_strerror(999) == "unknown error code"
    assert fa.fa_version() >= 100


def test_work_tiles_match_printed_table(lib):
    """Causal tiles computed: 36 of 64 at 1024 and 528 of 1024 at 4096 (block 128).

    fa_work_tiles walks one head's units through the kernel's own unit
    decoder (the loop bounds the forward kernel runs), not a closed form,
    so this pins the kernel's skip of future tiles."""
    rows = [line.split() for line in open(os.path.join(ROOT, "tests", "golden", "causal_tiles.txt"))
            if line.strip() and not line.startswith("#")]
    assert rows
    for ctx, block, computed, total, skipped in rows:
        assert int(block) == 128
        assert fa.fa_work_tiles(int(ctx), True) == int(computed)
        assert fa.fa_work_tiles(int(ctx), False) == int(total)
        assert round(100 * (1 - int(computed) / int(total))) == int(skipped)
    assert fa.fa_work_tiles(0, True) == 0
    assert fa.fa_work_tiles(129, True) == 3 and fa.fa_work_tiles(129, False) == 4
    # the closed forms n(n+1)/2 and n^2 (n = ceil(N/128)) for ragged and
    # odd tile counts, including a last unit whose second tile lies past N
    for n_tok in (1, 127, 128, 255, 256, 257, 383, 640, 1000, 8192, 32768):
        n = (n_tok + 127) // 128
        assert fa.fa_work_tiles(n_tok, True) == n * (n + 1) // 2
        assert fa.fa_work_tiles(n_tok, False) == n * n
    with pytest.raises(fa.FaError):
        fa.fa_work_tiles(-1, False)


FAKE = 0x10000  # 16-byte aligned, never dereferenced (errors are returned first)


def no_gpu():
    """Calls that pass every host check reach the device next; with FAKE
    pointers they are only made where there is no GPU to launch on."""
    import torch
    return not torch.cuda.is_available()


@pytest.mark.parametrize("args,code", [
    (dict(B=-1), fa.FA_ERR_SHAPE),
    (dict(N=-5), fa.FA_ERR_SHAPE),
    (dict(d=0), fa.FA_ERR_SHAPE),
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_SHAPE),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED_D),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED_D),
    (dict(dtype=7), fa.FA_ERR_DTYPE),
    (dict(scale=0.0), fa.FA_ERR_SCALE),
    (dict(scale=-1.0), fa.FA_ERR_SCALE),
    (dict(scale=float("nan")), fa.FA_ERR_SCALE),
    (dict(scale=float("inf")), fa.FA_ERR_SCALE),
    (dict(q=None), fa.FA_ERR_NULLPTR),
    (dict(lse=None), fa.FA_ERR_NULLPTR),
    (dict(k=FAKE + 8), fa.FA_ERR_ALIGN),
    (dict(o=FAKE + 2), fa.FA_ERR_ALIGN),
    (dict(lse=FAKE + 2), fa.FA_ERR_ALIGN),
    (dict(N=0, q=None, k=None, v=None, o=None, lse=None), fa.FA_OK),
    (dict(B=0), fa.FA_OK),
    (dict(H=0, q=None), fa.FA_OK),
])
def test_argument_errors(lib, args, code):
    call = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=2, N=300, d=128, causal=0,
                scale=0.125, dtype=fa.FA_BF16)
    call.update(args)
    assert fa.fa_fwd(**call) == code


def test_no_gpu_fails_loudly(lib):
    """Without a usable sm_103 device a valid call is refused, never computed on the CPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = fa.fa_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, 0, 0.125, fa.FA_FP16)
    assert rc == fa.FA_ERR_DEVICE
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fa.attention_forward(q, q, q)


def test_workspace_size_host_errors(lib):
    import ctypes as C
    out = C.c_size_t(7)
    assert lib.fa_fwd_workspace_size(1, 1, 256, 64, 0, None) == fa.FA_ERR_NULLPTR
    assert lib.fa_fwd_workspace_size(-1, 1, 256, 64, 0, C.byref(out)) == fa.FA_ERR_SHAPE
    assert lib.fa_fwd_workspace_size(1, 1, 256, 80, 0, C.byref(out)) == fa.FA_ERR_UNSUPPORTED_D
    assert lib.fa_fwd_workspace_size(0, 1, 256, 64, 0, C.byref(out)) == fa.FA_OK and out.value == 0
    # fa_fwd_ws validates like fa_fwd before touching the device
    assert fa.fa_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 300, 96, 0, 0.1, fa.FA_BF16,
                        None, 0) == fa.FA_ERR_UNSUPPORTED_D
    assert fa.fa_fwd_ws(None, FAKE, FAKE, FAKE, FAKE, 1, 1, 300, 64, 0, 0.1, fa.FA_BF16,
                        None, 0) == fa.FA_ERR_NULLPTR


def test_missing_library_raises(tmp_path):
    with pytest.raises(RuntimeError):
        fa.load_library(str(tmp_path / "libfa.so"))


def test_binding_dtype_contract():
    import torch
    assert fa.dtype_code(torch.bfloat16) == fa.FA_BF16
    assert fa.dtype_code(torch.float16) == fa.FA_FP16
    with pytest.raises(TypeError):
        fa.dtype_code(torch.float32)
    a = torch.zeros(1, 1, 4, 64, dtype=torch.float16)
    b = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fa.attention_forward(a, b, a)
    with pytest.raises(ValueError):
        fa.attention_forward(a[0], a[0], a[0])
    _ = ctypes  # keep the import used


def test_bwd_host_errors(lib):
    """fa_bwd checks its arguments before any device work, in fa_fwd's order."""
    call = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
                delta=FAKE, B=1, H=2, N=300, d=128, causal=1, scale=0.125, dtype=fa.FA_BF16)
    cases = [(dict(B=-1), fa.FA_ERR_SHAPE), (dict(d=80), fa.FA_ERR_UNSUPPORTED_D),
             (dict(dtype=3), fa.FA_ERR_DTYPE), (dict(scale=-2.0), fa.FA_ERR_SCALE),
             (dict(N=0, q=None), fa.FA_OK), (dict(dout=None), fa.FA_ERR_NULLPTR),
             (dict(delta=None), fa.FA_ERR_NULLPTR), (dict(dv=FAKE + 4), fa.FA_ERR_ALIGN),
             (dict(delta=FAKE + 2), fa.FA_ERR_ALIGN)]
    for args, code in cases:
        assert fa.fa_bwd(**{**call, **args}) == code, args
    import torch
    if not torch.cuda.is_available():
        assert fa.fa_bwd(**call) == fa.FA_ERR_DEVICE


def test_decode_host_errors(lib):
    """fa_decode checks shapes (1 <= Nq <= 16), width, dtype, scale, pointers."""
    call = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=2, H=4, Nq=1, Nk=5000, d=128,
                causal=0, scale=0.1, dtype=fa.FA_BF16, workspace=FAKE * 16, workspace_bytes=1 << 30)
    cases = [(dict(Nq=0), fa.FA_ERR_SHAPE), (dict(Nq=17), fa.FA_ERR_SHAPE),
             (dict(Nk=-1), fa.FA_ERR_SHAPE), (dict(d=32), fa.FA_ERR_UNSUPPORTED_D),
             (dict(dtype=9), fa.FA_ERR_DTYPE), (dict(scale=float("nan")), fa.FA_ERR_SCALE),
             (dict(B=0, q=None), fa.FA_OK), (dict(o=None), fa.FA_ERR_NULLPTR),
             (dict(k=None), fa.FA_ERR_NULLPTR), (dict(v=FAKE + 8), fa.FA_ERR_ALIGN)]
    for args, code in cases:
        assert fa.fa_decode(**{**call, **args}) == code, args
    import ctypes as C
    out = C.c_size_t(5)
    assert lib.fa_decode_workspace_size(1, 1, 17, 10, 64, C.byref(out)) == fa.FA_ERR_SHAPE
    assert lib.fa_decode_workspace_size(1, 1, 4, 0, 64, C.byref(out)) == fa.FA_OK and out.value == 0


def test_bwd_onepass_host_errors(lib):
    """fa_bwd_onepass checks fa_bwd's arguments, then its workspace, and
    only then reaches the device; its workspace is B*H*d*(N up to 128)*4."""
    import ctypes as C
    out = C.c_size_t(7)
    assert lib.fa_bwd_onepass_workspace_size(1, 1, 256, 64, None) == fa.FA_ERR_NULLPTR
    assert lib.fa_bwd_onepass_workspace_size(1, -1, 256, 64, C.byref(out)) == fa.FA_ERR_SHAPE
    assert lib.fa_bwd_onepass_workspace_size(1, 1, 256, 96, C.byref(out)) == fa.FA_ERR_UNSUPPORTED_D
    assert fa.fa_bwd_onepass_workspace_size(2, 3, 300, 128) == 2 * 3 * 128 * 384 * 4
    assert fa.fa_bwd_onepass_workspace_size(1, 1, 128, 64) == 64 * 128 * 4
    assert fa.fa_bwd_onepass_workspace_size(4, 4, 0, 64) == 0
    need = fa.fa_bwd_onepass_workspace_size(1, 2, 300, 64)
    call = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
                delta=FAKE, B=1, H=2, N=300, d=64, causal=1, scale=0.125, dtype=fa.FA_BF16,
                workspace=FAKE, workspace_bytes=need)
    for args, code in [(dict(d=96, workspace=None), fa.FA_ERR_UNSUPPORTED_D),
                       (dict(scale=0.0), fa.FA_ERR_SCALE),
                       (dict(dq=None), fa.FA_ERR_NULLPTR),
                       (dict(dk=FAKE + 4), fa.FA_ERR_ALIGN),
                       (dict(workspace=None), fa.FA_ERR_WORKSPACE),
                       (dict(workspace_bytes=need - 1), fa.FA_ERR_WORKSPACE),
                       (dict(workspace=FAKE + 8), fa.FA_ERR_ALIGN),
                       (dict(N=0, workspace=None), fa.FA_OK),
                       (dict(B=0, workspace=None), fa.FA_OK)]:
        assert fa.fa_bwd_onepass(**{**call, **args}) == code, args
    if no_gpu():
        assert fa.fa_bwd_onepass(**call) == fa.FA_ERR_DEVICE
    # the dropout form checks the probability first, then as fa_bwd_onepass
    dcall = {k: v for k, v in call.items() if k != "dtype"}
    dcall.update(dropout_p=0.1, seed=1, offset=2, dtype=fa.FA_BF16)
    assert fa.fa_bwd_onepass_dropout(**{**dcall, "dropout_p": 1.0, "d": 96}) == fa.FA_ERR_DROPOUT
    assert fa.fa_bwd_onepass_dropout(**{**dcall, "dropout_p": -0.1}) == fa.FA_ERR_DROPOUT
    assert fa.fa_bwd_onepass_dropout(**{**dcall, "d": 96}) == fa.FA_ERR_UNSUPPORTED_D
    assert fa.fa_bwd_onepass_dropout(**{**dcall, "workspace": None}) == fa.FA_ERR_WORKSPACE
    if no_gpu():
        assert fa.fa_bwd_onepass_dropout(**dcall) == fa.FA_ERR_DEVICE


def test_fwd_kv_host_errors(lib):
    """fa_fwd_kv checks shapes, the causal mode (0, 1, 2), widths, dtype, scale,
    pointers (k, v may be NULL only without keys) and alignment before the device."""
    call = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=2, H=4, Nq=300, Nk=5000, d=128,
                dv=64, causal=2, seqlens_k=None, scale=0.1, dtype=fa.FA_BF16)
    cases = [(dict(Nq=-1), fa.FA_ERR_SHAPE), (dict(Nk=-1), fa.FA_ERR_SHAPE),
             (dict(causal=3), fa.FA_ERR_SHAPE), (dict(causal=-1), fa.FA_ERR_SHAPE),
             (dict(d=96), fa.FA_ERR_UNSUPPORTED_D), (dict(dv=32), fa.FA_ERR_UNSUPPORTED_D),
             (dict(dv=0), fa.FA_ERR_SHAPE), (dict(dtype=7), fa.FA_ERR_DTYPE),
             (dict(scale=0.0), fa.FA_ERR_SCALE), (dict(Nq=0, q=None), fa.FA_OK),
             (dict(H=0), fa.FA_OK), (dict(o=None), fa.FA_ERR_NULLPTR),
             (dict(k=None), fa.FA_ERR_NULLPTR), (dict(q=FAKE + 4), fa.FA_ERR_ALIGN),
             (dict(seqlens_k=FAKE + 2), fa.FA_ERR_ALIGN)]
    for args, code in cases:
        assert fa.fa_fwd_kv(**{**call, **args}) == code, args
    # without keys, k and v may be NULL: the next check is the device's
    if no_gpu():
        rc = fa.fa_fwd_kv(**{**call, "Nk": 0, "k": None, "v": None})
        assert rc in (fa.FA_ERR_DEVICE, fa.FA_OK), rc


def test_fwd_varlen_host_errors(lib):
    """fa_fwd_varlen checks sizes, the causal mode, widths, dtype, scale,
    pointers (the offset arrays always; k, v only with keys) and alignment
    before the device."""
    call = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, cu_seqlens_q=FAKE, cu_seqlens_k=FAKE,
                B=3, H=4, max_seqlen_q=500, total_q=900, total_k=2000, d=64, dv=128, causal=1,
                scale=0.1, dtype=fa.FA_FP16)
    cases = [(dict(B=-1), fa.FA_ERR_SHAPE), (dict(total_k=-1), fa.FA_ERR_SHAPE),
             (dict(max_seqlen_q=-5), fa.FA_ERR_SHAPE), (dict(causal=7), fa.FA_ERR_SHAPE),
             (dict(d=32), fa.FA_ERR_UNSUPPORTED_D), (dict(dv=256), fa.FA_ERR_UNSUPPORTED_D),
             (dict(dtype=2), fa.FA_ERR_DTYPE), (dict(scale=float("inf")), fa.FA_ERR_SCALE),
             (dict(total_q=0, q=None), fa.FA_OK), (dict(max_seqlen_q=0), fa.FA_OK),
             (dict(B=0), fa.FA_OK), (dict(cu_seqlens_k=None), fa.FA_ERR_NULLPTR),
             (dict(v=None), fa.FA_ERR_NULLPTR), (dict(o=FAKE + 8), fa.FA_ERR_ALIGN),
             (dict(cu_seqlens_q=FAKE + 1), fa.FA_ERR_ALIGN),
             (dict(total_q=2 ** 30, H=4), fa.FA_ERR_SHAPE)]
    for args, code in cases:
        assert fa.fa_fwd_varlen(**{**call, **args}) == code, args
    if no_gpu():
        rc = fa.fa_fwd_varlen(**{**call, "total_k": 0, "k": None, "v": None})
        assert rc in (fa.FA_ERR_DEVICE, fa.FA_OK), rc


def test_unit_group_setter(lib):
    """fa_set_unit_group takes 0 (automatic) or a positive group size."""
    assert fa.fa_set_unit_group(-1) == fa.FA_ERR_SHAPE
    assert fa.fa_set_unit_group(4) == fa.FA_OK
    assert fa.fa_set_unit_group(0) == fa.FA_OK


def test_dropout_host_errors(lib):
    """fa_fwd_dropout / fa_bwd_dropout check the dropout probability (and
    the forward the causal mode) before anything else reaches the device."""
    fwd = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=2, N=300, d=64, causal=1,
               scale=0.125, dropout_p=0.1, seed=7, offset=0, dtype=fa.FA_BF16)
    for args, code in [(dict(dropout_p=1.0), fa.FA_ERR_DROPOUT),
                       (dict(dropout_p=-0.01), fa.FA_ERR_DROPOUT),
                       (dict(dropout_p=float("nan")), fa.FA_ERR_DROPOUT),
                       (dict(dropout_p=0.999), fa.FA_ERR_DROPOUT),
                       (dict(d=32), fa.FA_ERR_UNSUPPORTED_D),
                       (dict(o=None), fa.FA_ERR_NULLPTR), (dict(N=0), fa.FA_OK)]:
        assert fa.fa_fwd_dropout(**{**fwd, **args}) == code, args
    bwd = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
               delta=FAKE, B=1, H=2, N=300, d=128, causal=0, scale=0.1, dropout_p=0.3, seed=1,
               offset=5, dtype=fa.FA_FP16)
    for args, code in [(dict(dropout_p=1.5), fa.FA_ERR_DROPOUT), (dict(d=96), fa.FA_ERR_UNSUPPORTED_D),
                       (dict(delta=None), fa.FA_ERR_NULLPTR), (dict(B=0), fa.FA_OK)]:
        assert fa.fa_bwd_dropout(**{**bwd, **args}) == code, args
    assert "dropout" in fa.fa_strerror(fa.FA_ERR_DROPOUT)
    # the C entry point itself rejects a causal mode other than 0 or 1
    C = ctypes
    assert lib.fa_fwd_dropout(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 300, 64, 2, C.c_float(0.125),
                              C.c_float(0.1), 7, 0, fa.FA_BF16, None) == fa.FA_ERR_SHAPE


def test_bwd_kv_host_errors(lib):
    """fa_bwd_kv checks sizes, the causal mode (0 .. 2), width, dtype, scale,
    pointers (keys' only with keys, queries' only with queries) and
    alignment before the device."""
    call = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
                delta=FAKE, B=2, H=3, Nq=300, Nk=900, d=128, dv_width=64, causal=2, seqlens_k=None,
                scale=0.1, dtype=fa.FA_BF16)
    cases = [(dict(Nq=-1), fa.FA_ERR_SHAPE), (dict(causal=3), fa.FA_ERR_SHAPE),
             (dict(d=80), fa.FA_ERR_UNSUPPORTED_D), (dict(dv_width=96), fa.FA_ERR_UNSUPPORTED_D),
             (dict(dv_width=0), fa.FA_ERR_SHAPE), (dict(dtype=5), fa.FA_ERR_DTYPE),
             (dict(scale=-1.0), fa.FA_ERR_SCALE), (dict(Nq=0, Nk=0), fa.FA_OK), (dict(B=0), fa.FA_OK),
             (dict(dk=None), fa.FA_ERR_NULLPTR), (dict(delta=None), fa.FA_ERR_NULLPTR),
             (dict(seqlens_k=FAKE + 2), fa.FA_ERR_ALIGN), (dict(dq=FAKE + 8), fa.FA_ERR_ALIGN)]
    for args, code in cases:
        assert fa.fa_bwd_kv(**{**call, **args}) == code, args
    # without keys the key-side pointers, without queries the query-side
    # ones may be NULL: the next check is the device's
    for args in (dict(Nk=0, k=None, v=None, dk=None, dv=None),
                 dict(Nq=0, q=None, o=None, dout=None, dq=None, lse=None, delta=None)):
        if no_gpu():
            assert fa.fa_bwd_kv(**{**call, **args}) in (fa.FA_ERR_DEVICE, fa.FA_OK), args
    # the square entry point keeps its causal contract (0 or 1)
    C = ctypes
    assert lib.fa_bwd(*([FAKE] * 10), 1, 2, 256, 64, 2, C.c_float(0.125), fa.FA_BF16,
                      None) == fa.FA_ERR_SHAPE


def test_bwd_varlen_host_errors(lib):
    """fa_bwd_varlen checks sizes, causal mode, width, dtype, scale, the
    offset arrays and the other pointers, and alignment before the device."""
    call = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
                delta=FAKE, cu_seqlens_q=FAKE, cu_seqlens_k=FAKE, B=3, H=2, max_seqlen_q=500,
                max_seqlen_k=700, total_q=900, total_k=1500, d=64, dv_width=128, causal=1,
                scale=0.125, dtype=fa.FA_FP16)
    cases = [(dict(total_k=-1), fa.FA_ERR_SHAPE), (dict(max_seqlen_k=-1), fa.FA_ERR_SHAPE),
             (dict(causal=3), fa.FA_ERR_SHAPE), (dict(d=32), fa.FA_ERR_UNSUPPORTED_D),
             (dict(dv_width=80), fa.FA_ERR_UNSUPPORTED_D),
             (dict(dtype=9), fa.FA_ERR_DTYPE), (dict(scale=0.0), fa.FA_ERR_SCALE),
             (dict(B=0), fa.FA_OK), (dict(total_q=0, total_k=0), fa.FA_OK),
             (dict(cu_seqlens_k=None), fa.FA_ERR_NULLPTR), (dict(dv=None), fa.FA_ERR_NULLPTR),
             (dict(delta=FAKE + 2), fa.FA_ERR_ALIGN), (dict(k=FAKE + 8), fa.FA_ERR_ALIGN)]
    for args, code in cases:
        assert fa.fa_bwd_varlen(**{**call, **args}) == code, args
    if no_gpu():
        assert fa.fa_bwd_varlen(**call) in (fa.FA_ERR_DEVICE, fa.FA_OK)


def test_watchdog_selftest_host_errors(lib):
    assert fa.fa_watchdog_selftest(0) == fa.FA_ERR_SHAPE
    assert fa.fa_watchdog_selftest(10 ** 10) == fa.FA_ERR_SHAPE
    import torch
    if not torch.cuda.is_available():
        assert fa.fa_watchdog_selftest(1000) == fa.FA_ERR_DEVICE


def test_kv_varlen_dropout_host_errors(lib):
    """The dropout forms of the kv and packed-batch entry points check the
    dropout probability first, then the arguments of their plain forms, and
    only then reach the device."""
    kv = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=2, H=4, Nq=300, Nk=5000, d=128, dv=64,
              causal=2, seqlens_k=None, scale=0.1, dropout_p=0.2, seed=3, offset=1,
              dtype=fa.FA_BF16)
    vl = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, cu_seqlens_q=FAKE, cu_seqlens_k=FAKE, B=3,
              H=4, max_seqlen_q=500, total_q=900, total_k=2000, d=64, dv=128, causal=1, scale=0.1,
              dropout_p=0.2, seed=3, offset=1, dtype=fa.FA_FP16)
    bkv = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
               delta=FAKE, B=2, H=3, Nq=300, Nk=900, d=128, dv_width=64, causal=2, seqlens_k=None,
               scale=0.1, dropout_p=0.2, seed=3, offset=1, dtype=fa.FA_BF16)
    bvl = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
               delta=FAKE, cu_seqlens_q=FAKE, cu_seqlens_k=FAKE, B=3, H=4, max_seqlen_q=500,
               max_seqlen_k=2000, total_q=900, total_k=2000, d=64, dv_width=128, causal=1,
               scale=0.1, dropout_p=0.2, seed=3, offset=1, dtype=fa.FA_FP16)
    for fn, base, bad_shape in [(fa.fa_fwd_kv_dropout, kv, dict(causal=3)),
                                (fa.fa_fwd_varlen_dropout, vl, dict(causal=7)),
                                (fa.fa_bwd_kv_dropout, bkv, dict(causal=3)),
                                (fa.fa_bwd_varlen_dropout, bvl, dict(causal=7))]:
        for args, code in [(dict(dropout_p=1.0), fa.FA_ERR_DROPOUT),
                           (dict(dropout_p=-0.5), fa.FA_ERR_DROPOUT),
                           (dict(dropout_p=float("nan")), fa.FA_ERR_DROPOUT),
                           (dict(dropout_p=0.999, d=96), fa.FA_ERR_DROPOUT),
                           (dict(d=96), fa.FA_ERR_UNSUPPORTED_D), (bad_shape, fa.FA_ERR_SHAPE),
                           (dict(dtype=9), fa.FA_ERR_DTYPE), (dict(scale=0.0), fa.FA_ERR_SCALE),
                           (dict(o=None), fa.FA_ERR_NULLPTR), (dict(B=0), fa.FA_OK)]:
            assert fn(**{**base, **args}) == code, (fn.__name__, args)
        # p = 0 and p > 0 both pass the host checks; the next check is the device's
        if no_gpu():
            for p_ in (0.0, 0.25):
                assert fn(**{**base, "dropout_p": p_}) in (fa.FA_ERR_DEVICE, fa.FA_OK), fn.__name__
