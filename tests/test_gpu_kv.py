"""fa_fwd_kv (queries against a key set of another length, per-batch key
counts, explicit causal alignment) vs the float64 oracle, through the C ABI.

The oracle gets each (batch, head) with its keys cut to the batch's count
and every query row at its absolute position (row i at i for upper-left,
at len_b - Nq + i for bottom-right), so alignment and padding are checked
against the plain definition; a row with no visible key must come back as
O = 0 and LSE = -inf exactly (the pages' policy for an empty key set).
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import oracle
import seeded_inputs
from gpu_common import LSE_TOL, TOL, default_scale, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_kv(q, k, v, causal, seqlens, scale):
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    sl = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    o, lse = fa.attention_forward_kv(dq, dk, dv, causal=causal, seqlens_k=sl, scale=scale)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    return o.cpu(), lse.cpu()


def oracle_kv(q, k, v, causal, seqlens, scale):
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    o = np.zeros((B, H, Nq, v.shape[3]))
    lse = np.zeros((B, H, Nq))
    for b in range(B):
        n = Nk if seqlens is None else max(0, min(seqlens[b], Nk))
        pos = np.arange(Nq, dtype=np.int64)
        if causal == "bottom_right":
            pos = pos + (n - Nq)
        for h in range(H):
            ob, lb = oracle.attention_rows(q[b, h].double().numpy(), pos,
                                           k[b, h, :n].double().numpy(), v[b, h, :n].double().numpy(),
                                           causal=causal is not None, scale=scale)
            o[b, h], lse[b, h] = ob, lb
    return o, lse


def check(o, lse, o_ref, lse_ref, dtype, what):
    o = o.double().numpy()
    lse = lse.double().numpy()
    empty = np.isneginf(lse_ref)
    # rows that see no key: exactly O = 0 and LSE = -inf
    assert np.all(np.isneginf(lse[empty])), f"{what}: empty rows must have LSE = -inf"
    assert np.all(o[empty] == 0.0), f"{what}: empty rows must have O = 0"
    full = ~empty
    assert np.all(np.isfinite(lse[full])) and np.all(np.isfinite(o)), f"{what}: non-finite values"
    if not full.any():
        return
    err = np.abs(o[full] - o_ref[full])
    tmax, tmean = TOL[dtype]
    assert err.max() <= tmax, f"{what}: max|dO| {err.max():.3e}"
    assert err.mean() <= tmean, f"{what}: mean|dO| {err.mean():.3e}"
    lerr = np.abs(lse[full] - lse_ref[full]).max()
    assert lerr <= LSE_TOL, f"{what}: max|dLSE| {lerr:.3e}"


CASES = [
    # B, H, Nq, Nk, d, dtype, causal, seqlens
    (1, 2, 200, 1000, 64, "bf16", "bottom_right", None),       # prefill chunk after a cache
    (2, 2, 333, 777, 128, "fp16", "upper_left", None),
    (2, 1, 300, 128, 64, "fp16", "bottom_right", None),        # Nq > Nk: the first rows see nothing
    (1, 2, 100, 50, 128, "bf16", "upper_left", None),          # Nq > Nk, every row sees key 0
    (3, 2, 256, 1024, 128, "bf16", None, [1024, 500, 0]),      # padding, one empty batch
    (3, 1, 129, 700, 64, "bf16", "bottom_right", [700, 64, 1]),
    (2, 2, 260, 900, 64, "fp16", "upper_left", [900, 131]),
    (1, 1, 1, 5000, 64, "fp16", "bottom_right", None),         # one query against a long cache
    (1, 3, 7, 3, 128, "fp16", None, None),
    (2, 1, 640, 2000, 128, "bf16", "bottom_right", [2000, 1500]),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,causal,seqlens", CASES,
                         ids=[f"B{c[0]}H{c[1]}q{c[2]}k{c[3]}d{c[4]}{c[5]}{c[6] or 'nc'}"
                              f"{'' if c[7] is None else 'pad'}" for c in CASES])
def test_kv_vs_oracle(B, H, Nq, Nk, d, dtype, causal, seqlens):
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, dtype, seed=Nq + 3 * Nk + d)
    scale = default_scale(d)
    o, lse = run_kv(q, k, v, causal, seqlens, scale)
    o_ref, lse_ref = oracle_kv(q, k, v, causal, seqlens, scale)
    check(o, lse, o_ref, lse_ref, dtype, f"B{B}H{H}q{Nq}k{Nk}d{d}{dtype}{causal}{seqlens}")


@pytest.mark.parametrize("d,dtype,causal", [(64, "bf16", False), (128, "fp16", True),
                                            (64, "fp16", True), (128, "bf16", False)])
def test_square_equals_fa_fwd(d, dtype, causal):
    """Nq = Nk, all keys, upper-left: the same tiles in the same order as fa_fwd."""
    q, k, v = seeded_inputs.make_qkv(2, 2, 600, d, dtype, 1.5, seed=31 + d)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    o1, l1 = fa.attention_forward(dq, dk, dv, causal=causal)
    o2, l2 = fa.attention_forward_kv(dq, dk, dv, causal="upper_left" if causal else None)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


DV_CASES = [
    # B, H, Nq, Nk, d, dv, dtype, causal, seqlens
    (1, 2, 300, 700, 64, 128, "bf16", "bottom_right", None),
    (2, 1, 257, 257, 128, 64, "fp16", "upper_left", None),
    (2, 2, 200, 1000, 128, 64, "bf16", None, [1000, 333]),
    (1, 1, 129, 64, 64, 128, "fp16", "bottom_right", None),     # first rows see nothing
    (1, 3, 640, 640, 64, 128, "fp16", None, None),
    (2, 1, 1, 3000, 128, 64, "bf16", "bottom_right", [3000, 17]),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,dtype,causal,seqlens", DV_CASES,
                         ids=[f"B{c[0]}H{c[1]}q{c[2]}k{c[3]}d{c[4]}dv{c[5]}{c[6]}{c[7] or 'nc'}"
                              for c in DV_CASES])
def test_value_width_vs_oracle(B, H, Nq, Nk, d, dv, dtype, causal, seqlens):
    """A value width dv different from the query/key width d (the pages'
    reference allows it and tests it): O is [B, H, Nq, dv]."""
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, dtype, seed=7 * Nq + Nk + dv, dv=dv)
    scale = default_scale(d)
    o, lse = run_kv(q, k, v, causal, seqlens, scale)
    assert o.shape == (B, H, Nq, dv)
    o_ref, lse_ref = oracle_kv(q, k, v, causal, seqlens, scale)
    check(o, lse, o_ref, lse_ref, dtype, f"B{B}H{H}q{Nq}k{Nk}d{d}dv{dv}{dtype}{causal}{seqlens}")


def test_value_width_guard_columns():
    """With dv = 64 < d = 128 the kernel must write exactly dv columns per
    row: a guard band around O stays untouched."""
    B, H, Nq, Nk, d, dv = 1, 2, 300, 400, 128, 64
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, "bf16", seed=77, dv=dv)
    dq, dk, dvv = (t.cuda() for t in (q, k, v))
    n = B * H * Nq * dv
    buf = torch.full((n + 2 * 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    o = buf[4096:4096 + n].view(B, H, Nq, dv)
    fa.attention_forward_kv(dq, dk, dvv, causal="bottom_right", out=o)
    torch.cuda.synchronize()
    assert torch.all(buf[:4096] == 7.0) and torch.all(buf[4096 + n:] == 7.0)
    o_ref, _ = oracle_kv(q, k, v, "bottom_right", None, default_scale(d))
    assert np.abs(o.cpu().double().numpy() - o_ref).max() <= TOL["bf16"][0]


def test_no_keys():
    """Nk = 0, and every batch padded to zero keys: O = 0, LSE = -inf."""
    q, k, v = seeded_inputs.make_decode(2, 2, 150, 1, 64, "bf16", seed=5)
    dq = q.cuda()
    o, lse = fa.attention_forward_kv(dq, k[:, :, :0].cuda().contiguous(),
                                     v[:, :, :0].cuda().contiguous(), causal="bottom_right")
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    dk, dv = k.cuda(), v.cuda()
    sl = torch.zeros(2, dtype=torch.int32, device="cuda")
    o, lse = fa.attention_forward_kv(dq, dk, dv, causal=None, seqlens_k=sl)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    assert fa.fa_status()[0] == fa.FA_OK


def test_errors():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 128, dtype=torch.float32, device="cuda")
    s = 0.125
    assert fa.fa_fwd_kv(q, q, q, o, lse, 1, 1, 128, 128, 64, 64, 3, None, s, fa.FA_BF16) == fa.FA_ERR_SHAPE
    assert fa.fa_fwd_kv(q, q, q, o, lse, 1, 1, 128, -1, 64, 64, 0, None, s, fa.FA_BF16) == fa.FA_ERR_SHAPE
    sl = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert fa.fa_fwd_kv(q, q, q, o, lse, 1, 1, 128, 128, 64, 64, 1, sl.data_ptr() + 2, s,
                        fa.FA_BF16) == fa.FA_ERR_ALIGN
    assert fa.fa_fwd_kv(q, q, q, o, lse, 1, 1, 0, 128, 64, 64, 1, None, s, fa.FA_BF16) == fa.FA_OK
    assert fa.fa_fwd_kv(q, q, q, o, lse, 1, 1, 128, 128, 64, 96, 0, None, s,
                        fa.FA_BF16) == fa.FA_ERR_UNSUPPORTED_D
