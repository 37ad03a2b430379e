"""fa_fwd_dropout / fa_bwd_dropout vs the float64 dropout oracle, through the
C ABI.

The kernels draw the mask on the device from (seed, offset) and never store
it; the oracle draws the same mask from its own implementation of the same
generator (each head with its batch*head index), so every row of O, LSE,
dQ, dK and dV is checked against the plain definition with that mask.  The
backward pass regenerating the forward's mask is what the pages keep the
generator state for ("Why FlashAttention Can Avoid a Square Attention Array
Without Making Attention Linear", section "Backward can recreate tiles
instead of retaining the square").
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import oracle
import seeded_inputs
from gpu_common import LSE_TOL, TOL, default_scale, require_gpu
from test_gpu_backward import check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


CASES = [
    # B, H, N, d, dtype, causal, p, seed, offset
    (1, 2, 300, 64, "bf16", True, 0.1, 1234, 0),
    (2, 1, 257, 128, "fp16", False, 0.5, 7, 3),
    (1, 1, 129, 128, "bf16", True, 0.3, 2 ** 40 + 3, 11),
    (1, 2, 640, 64, "fp16", False, 0.2, 99, 2 ** 31 + 5),
    (1, 1, 1, 64, "bf16", True, 0.6, 5, 0),
]


def ids(c):
    return f"B{c[0]}H{c[1]}N{c[2]}d{c[3]}{c[4]}{'c' if c[5] else 'nc'}p{c[6]}"


def oracle_fwd(q, k, v, causal, p, seed, off, scale):
    B, H, N, d = q.shape
    o, lse = np.zeros(q.shape), np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = oracle.attention_dropout(q[b, h], k[b, h], v[b, h], b * H + h, seed,
                                                          off, p, causal=causal, scale=scale)
    return o, lse


@pytest.mark.parametrize("B,H,N,d,dtype,causal,p,seed,off", CASES, ids=[ids(c) for c in CASES])
def test_forward_dropout_vs_oracle(B, H, N, d, dtype, causal, p, seed, off):
    q, k, v = seeded_inputs.make_qkv(B, H, N, d, dtype, 1.0, seed=N + d)
    scale = default_scale(d)
    o, lse = fa.attention_forward_dropout(q.cuda(), k.cuda(), v.cuda(), p, seed, off, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_status()[0] == fa.FA_OK
    o_ref, lse_ref = oracle_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), causal,
                                p, seed, off, scale)
    # Kept weights are scaled by s = 256 / t, so O and its rounding errors (P
    # to 16 bits, the final rounding of O) grow by s: the absolute bounds on
    # O are the forward's times s; LSE does not depend on dropout.
    s = 256.0 / oracle.dropout_threshold(p)
    o = o.cpu().double().numpy()
    what = ids((B, H, N, d, dtype, causal, p))
    assert np.all(np.isfinite(o)), what
    err = np.abs(o - o_ref)
    tmax, tmean = TOL[dtype]
    assert err.max() <= tmax * s, f"{what}: max|dO| {err.max():.3e} > {tmax * s:.3e}"
    assert err.mean() <= tmean * s, f"{what}: mean|dO| {err.mean():.3e} > {tmean * s:.3e}"
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= LSE_TOL, what


@pytest.mark.parametrize("B,H,N,d,dtype,causal,p,seed,off", CASES[:4], ids=[ids(c) for c in CASES[:4]])
def test_backward_dropout_vs_oracle(B, H, N, d, dtype, causal, p, seed, off):
    q, k, v = seeded_inputs.make_qkv(B, H, N, d, dtype, 1.0, seed=N + d)
    dout = seeded_inputs.make_dout(B, H, N, d, dtype, seed=N + d)
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    o, lse = fa.attention_forward_dropout(dq_, dk_, dv_, p, seed, off, causal=causal)
    gq, gk, gv = fa.attention_backward_dropout(dq_, dk_, dv_, o, lse, do_, p, seed, off,
                                               causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_status()[0] == fa.FA_OK
    scale = default_scale(d)
    rq, rk, rv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            rq[b, h], rk[b, h], rv[b, h] = oracle.attention_dropout_grad(
                q[b, h].double().numpy(), k[b, h].double().numpy(), v[b, h].double().numpy(),
                dout[b, h].double().numpy(), b * H + h, seed, off, p, causal=causal, scale=scale)
    name = ids((B, H, N, d, dtype, causal, p))
    check_grad(name + " dQ", gq.cpu(), rq, dtype)
    check_grad(name + " dK", gk.cpu(), rk, dtype)
    check_grad(name + " dV", gv.cpu(), rv, dtype)


def test_zero_probability_is_fa_fwd():
    q, k, v = (t.cuda() for t in seeded_inputs.make_qkv(1, 3, 400, 128, "bf16", 1.0, seed=2))
    o1, l1 = fa.attention_forward(q, k, v, causal=True)
    o2, l2 = fa.attention_forward_dropout(q, k, v, 0.0, 123, 4, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_mask_follows_seed_and_offset():
    """The same (seed, offset) gives the same output; another offset or seed
    another mask; LSE never depends on the mask."""
    q, k, v = (t.cuda() for t in seeded_inputs.make_qkv(1, 2, 300, 64, "fp16", 1.0, seed=3))
    a, la = fa.attention_forward_dropout(q, k, v, 0.25, 10, 0)
    b, lb = fa.attention_forward_dropout(q, k, v, 0.25, 10, 0)
    c, lc = fa.attention_forward_dropout(q, k, v, 0.25, 10, 1)
    e, le = fa.attention_forward_dropout(q, k, v, 0.25, 11, 0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, e)
    assert torch.equal(la, lc) and torch.equal(la, le)


def test_dropout_errors():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError):
        fa.attention_forward_dropout(q, q, q, 1.0, 0, 0)
    with pytest.raises(fa.FaError):
        fa.attention_forward_dropout(q, q, q, -0.5, 0, 0)
