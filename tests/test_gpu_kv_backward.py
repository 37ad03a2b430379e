"""fa_bwd_kv (the backward pass of fa_fwd_kv: queries against a key set of
another length, per-batch key counts, explicit causal alignment) vs the
float64 gradient oracle, through the C ABI.

The oracle gets each (batch, head) with its keys cut to the batch's count:
dQ (with the row's LSE and D) at every query's absolute position, then dK
and dV of those keys with their positions shifted by the query offset
(key j is visible to query i iff j <= i + off, i.e. j - off <= i).  Keys
past a batch's count must come back with dK = dV = 0 exactly, and query
rows that see no key with dQ = 0.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import oracle
import seeded_inputs
from gpu_common import default_scale, require_gpu
from test_gpu_backward import check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def oracle_kv_grad(q, k, v, dout, causal, seqlens, scale):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    gq, gk, gv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(B):
        n = Nk if seqlens is None else max(0, min(seqlens[b], Nk))
        off = n - Nq if causal == "bottom_right" else 0
        pos = np.arange(Nq, dtype=np.int64) + off
        for h in range(H):
            qh, gh = q[b, h].double().numpy(), dout[b, h].double().numpy()
            kh, vh = k[b, h, :n].double().numpy(), v[b, h, :n].double().numpy()
            dq, lse, delta = oracle.grad_query_rows(qh, gh, pos, kh, vh, causal=causal is not None,
                                                    scale=scale)
            gq[b, h] = dq
            if n:
                dk, dv = oracle.grad_key_rows(kh, vh, np.arange(n, dtype=np.int64) - off, qh, gh,
                                              lse, delta, causal=causal is not None, scale=scale)
                gk[b, h, :n], gv[b, h, :n] = dk, dv
    return gq, gk, gv


def run_kv_bwd(q, k, v, dout, causal, seqlens, scale):
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    sl = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    o, lse = fa.attention_forward_kv(dq_, dk_, dv_, causal=causal, seqlens_k=sl, scale=scale)
    g = fa.attention_backward_kv(dq_, dk_, dv_, o, lse, do_, causal=causal, seqlens_k=sl,
                                 scale=scale)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    return tuple(t.cpu() for t in g)


CASES = [
    # B, H, Nq, Nk, d, dtype, causal, seqlens
    (1, 2, 200, 1000, 64, "bf16", "bottom_right", None),       # a chunk after a cache
    (2, 1, 333, 777, 128, "fp16", "upper_left", None),
    (2, 1, 300, 128, 64, "fp16", "bottom_right", None),        # Nq > Nk: the first rows see nothing
    (3, 2, 256, 1024, 128, "bf16", None, [1024, 500, 0]),      # padding, one empty batch
    (3, 1, 129, 700, 64, "bf16", "bottom_right", [700, 64, 1]),
    (2, 2, 260, 900, 64, "fp16", "upper_left", [900, 131]),
    (1, 1, 640, 2000, 128, "bf16", "bottom_right", [1500]),
    # ten (batch, head) pairs: work items dealt in groups of 8 heads, the
    # last group of 2
    (5, 2, 200, 600, 64, "bf16", "bottom_right", [600, 300, 0, 129, 450]),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,causal,seqlens", CASES,
                         ids=[f"B{c[0]}H{c[1]}q{c[2]}k{c[3]}d{c[4]}{c[5]}{c[6] or 'nc'}"
                              f"{'' if c[7] is None else 'pad'}" for c in CASES])
def test_kv_backward_vs_oracle(B, H, Nq, Nk, d, dtype, causal, seqlens):
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, dtype, seed=Nq + 5 * Nk + d)
    dout = seeded_inputs.make_dout(B, H, Nq, d, dtype, seed=Nq + Nk)
    scale = default_scale(d)
    gq, gk, gv = run_kv_bwd(q, k, v, dout, causal, seqlens, scale)
    rq, rk, rv = oracle_kv_grad(q, k, v, dout, causal, seqlens, scale)
    name = f"B{B}H{H}q{Nq}k{Nk}d{d}{dtype}{causal}{seqlens}"
    check_grad(name + " dQ", gq, rq, dtype)
    check_grad(name + " dK", gk, rk, dtype)
    check_grad(name + " dV", gv, rv, dtype)
    # padded keys and rows that see nothing are exactly zero
    for b in range(B):
        n = Nk if seqlens is None else max(0, min(seqlens[b], Nk))
        assert torch.all(gk[b, :, n:] == 0) and torch.all(gv[b, :, n:] == 0)
        if n == 0:
            assert torch.all(gq[b] == 0)


WIDTH_CASES = [
    # B, H, Nq, Nk, d, dv, dtype, causal, seqlens
    (1, 2, 200, 1000, 64, 128, "bf16", "bottom_right", None),    # a chunk after a cache
    (2, 1, 333, 777, 128, 64, "fp16", "upper_left", None),
    (3, 1, 256, 700, 128, 64, "bf16", None, [700, 100, 0]),       # padding, one empty batch
    (1, 1, 300, 128, 64, 128, "fp16", "bottom_right", None),     # Nq > Nk: rows that see nothing
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,dtype,causal,seqlens", WIDTH_CASES,
                         ids=[f"B{c[0]}H{c[1]}q{c[2]}k{c[3]}d{c[4]}dv{c[5]}{c[6]}{c[7] or 'nc'}"
                              f"{'' if c[8] is None else 'pad'}" for c in WIDTH_CASES])
def test_kv_backward_value_width(B, H, Nq, Nk, d, dv, dtype, causal, seqlens):
    """Values (and O, dO, dV) of another width than queries and keys: the
    kernels load each tensor at its own width, take d / 16 or dv / 16 K
    steps and accumulate dV over dv columns, dK and dQ over d."""
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, dtype, seed=Nq + 5 * Nk + d + dv, dv=dv)
    dout = seeded_inputs.make_dout(B, H, Nq, dv, dtype, seed=Nq + Nk + dv)
    scale = default_scale(d)
    gq, gk, gv = run_kv_bwd(q, k, v, dout, causal, seqlens, scale)
    assert gq.shape == q.shape and gk.shape == k.shape and gv.shape == v.shape
    rq, rk, rv = oracle_kv_grad(q, k, v, dout, causal, seqlens, scale)
    name = f"B{B}H{H}q{Nq}k{Nk}d{d}dv{dv}{dtype}{causal}{seqlens}"
    check_grad(name + " dQ", gq, rq, dtype)
    check_grad(name + " dK", gk, rk, dtype)
    check_grad(name + " dV", gv, rv, dtype)
    for b in range(B):
        n = Nk if seqlens is None else max(0, min(seqlens[b], Nk))
        assert torch.all(gk[b, :, n:] == 0) and torch.all(gv[b, :, n:] == 0)


@pytest.mark.parametrize("d,dtype,causal", [(64, "bf16", True), (128, "fp16", False)])
def test_square_equals_fa_bwd(d, dtype, causal):
    """Nq = Nk, all keys, upper-left: the same tiles and masks as fa_bwd."""
    q, k, v = (t.cuda() for t in seeded_inputs.make_qkv(2, 2, 600, d, dtype, 1.0, seed=17 + d))
    do = seeded_inputs.make_dout(2, 2, 600, d, dtype, seed=17).cuda()
    o, lse = fa.attention_forward(q, k, v, causal=causal)
    g1 = fa.attention_backward(q, k, v, o, lse, do, causal=causal)
    g2 = fa.attention_backward_kv(q, k, v, o, lse, do, causal="upper_left" if causal else None)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_kv_backward_without_queries_or_keys():
    q, k, v = seeded_inputs.make_decode(2, 2, 150, 300, 64, "bf16", seed=8)
    dq_, dk_, dv_ = q.cuda(), k.cuda(), v.cuda()
    do_ = seeded_inputs.make_dout(2, 2, 150, 64, "bf16", seed=8).cuda()
    # no keys at all: every dQ row is zero
    k0, v0 = dk_[:, :, :0].contiguous(), dv_[:, :, :0].contiguous()
    o, lse = fa.attention_forward_kv(dq_, k0, v0, causal="bottom_right")
    gq, gk, gv = fa.attention_backward_kv(dq_, k0, v0, o, lse, do_, causal="bottom_right")
    torch.cuda.synchronize()
    assert torch.all(gq == 0) and gk.numel() == 0
    # no queries: every dK, dV row is zero
    q0, d0 = dq_[:, :, :0].contiguous(), do_[:, :, :0].contiguous()
    o, lse = fa.attention_forward_kv(q0, dk_, dv_, causal=None)
    gq, gk, gv = fa.attention_backward_kv(q0, dk_, dv_, o, lse, d0, causal=None)
    torch.cuda.synchronize()
    assert gq.numel() == 0 and torch.all(gk == 0) and torch.all(gv == 0)
    assert fa.fa_status()[0] == fa.FA_OK


def test_kv_backward_errors():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    assert fa.fa_bwd_kv(q, q, q, q, lse, q, q, q, q, lse, 1, 1, 128, 128, 64, 64, 3, None, 0.125,
                        fa.FA_BF16) == fa.FA_ERR_SHAPE
    assert fa.fa_bwd_kv(q, q, q, q, lse, q, q, q, q, lse, 1, 1, 128, 128, 96, 64, 0, None, 0.125,
                        fa.FA_BF16) == fa.FA_ERR_UNSUPPORTED_D
    assert fa.fa_bwd_kv(q, q, q, q, lse, q, q, q, q, lse, 1, 1, 128, 128, 64, 32, 0, None, 0.125,
                        fa.FA_BF16) == fa.FA_ERR_UNSUPPORTED_D
