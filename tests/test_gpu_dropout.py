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


# ---------------------------------------------------------------- kv and packed batches

KV_CASES = [
    # B, H, Nq, Nk, d, dv, dtype, causal, seqlens, p
    (2, 1, 200, 700, 64, 64, "bf16", "bottom_right", None, 0.2),      # a chunk after a cache
    (3, 2, 256, 500, 128, 64, "fp16", None, [500, 130, 0], 0.1),       # padding, an empty batch
    (1, 1, 300, 128, 64, 128, "bf16", "bottom_right", None, 0.3),     # Nq > Nk: empty rows
    (2, 1, 333, 777, 128, 128, "fp16", "upper_left", [777, 400], 0.5),
]


def kv_ids(c):
    return (f"B{c[0]}H{c[1]}q{c[2]}k{c[3]}d{c[4]}dv{c[5]}{c[6]}{c[7] or 'nc'}"
            f"{'' if c[8] is None else 'pad'}p{c[9]}")


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,dtype,causal,seqlens,p", KV_CASES,
                         ids=[kv_ids(c) for c in KV_CASES])
def test_kv_dropout_vs_oracle(B, H, Nq, Nk, d, dv, dtype, causal, seqlens, p):
    """fa_fwd_kv_dropout / fa_bwd_kv_dropout against the dropout oracle run per
    (batch, head) on the batch's keys, each query at its row's position (the
    mask indexed by row and key, the alignment moving only the causal
    boundary); rows that see no key come back as O = 0, LSE = -inf, keys no
    query sees as dK = dV = 0."""
    seed, off = 4242 + Nq, 6
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, dtype, seed=Nq + Nk + dv, dv=dv)
    dout = seeded_inputs.make_dout(B, H, Nq, dv, dtype, seed=Nq + dv)
    scale = default_scale(d)
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    sl = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    o, lse = fa.attention_forward_kv(dq_, dk_, dv_, causal=causal, seqlens_k=sl, scale=scale,
                                     dropout_p=p, seed=seed, offset=off)
    gq, gk, gv = fa.attention_backward_kv(dq_, dk_, dv_, o, lse, do_, causal=causal, seqlens_k=sl,
                                          scale=scale, dropout_p=p, seed=seed, offset=off)
    torch.cuda.synchronize()
    assert fa.fa_status()[0] == fa.FA_OK
    o, lse, gq, gk, gv = (t.cpu() for t in (o, lse, gq, gk, gv))
    s = 256.0 / oracle.dropout_threshold(p)
    tmax, tmean = TOL[dtype]
    rq, rk, rv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for b in range(B):
        n = Nk if seqlens is None else max(0, min(seqlens[b], Nk))
        shift = n - Nq if causal == "bottom_right" else 0
        for h in range(H):
            args = (q[b, h].double().numpy(), k[b, h, :n].double().numpy(),
                    v[b, h, :n].double().numpy())
            o_ref, l_ref = oracle.attention_dropout(*args, b * H + h, seed, off, p,
                                                    causal=causal is not None, scale=scale,
                                                    q_offset=shift)
            ob, lb = o[b, h].double().numpy(), lse[b, h].double().numpy()
            empty = np.isneginf(l_ref)
            assert np.all(np.isneginf(lb[empty])) and np.all(ob[empty] == 0.0)
            err = np.abs(ob[~empty] - o_ref[~empty])
            if err.size:
                assert err.max() <= tmax * s and err.mean() <= tmean * s, (b, h, err.max())
                assert np.abs(lb[~empty] - l_ref[~empty]).max() <= LSE_TOL
            gq_r, gk_r, gv_r = oracle.attention_dropout_grad(
                *args, dout[b, h].double().numpy(), b * H + h, seed, off, p,
                causal=causal is not None, scale=scale, q_offset=shift)
            rq[b, h], rk[b, h, :n], rv[b, h, :n] = gq_r, gk_r, gv_r
        assert torch.all(gk[b, :, n:] == 0) and torch.all(gv[b, :, n:] == 0)
    name = kv_ids((B, H, Nq, Nk, d, dv, dtype, causal, seqlens, p))
    check_grad(name + " dQ", gq, rq, dtype)
    check_grad(name + " dK", gk, rk, dtype)
    check_grad(name + " dV", gv, rv, dtype)


VARLEN_CASES = [
    # name, lens_q, lens_k, H, d, dv, dtype, causal, p
    ("self_ul", [1, 127, 129, 300, 0, 517], [1, 127, 129, 300, 0, 517], 2, 64, 64, "bf16",
     "upper_left", 0.2),
    ("prefill_br", [64, 200, 1], [1000, 250, 3000], 2, 128, 64, "fp16", "bottom_right", 0.1),
]


@pytest.mark.parametrize("name,lens_q,lens_k,H,d,dv,dtype,causal,p", VARLEN_CASES,
                         ids=[c[0] for c in VARLEN_CASES])
def test_varlen_dropout_vs_oracle(name, lens_q, lens_k, H, d, dv, dtype, causal, p):
    """fa_fwd_varlen_dropout / fa_bwd_varlen_dropout against the dropout oracle
    run per (sequence, head), the mask of sequence b's head h drawn with
    index b * H + h."""
    seed, off = 31337, 2
    q, k, v, cu_q, cu_k = seeded_inputs.make_varlen(lens_q, lens_k, H, d, dtype, seed=len(lens_q) + dv,
                                                    dv=dv)
    g = torch.Generator("cpu").manual_seed(len(lens_q) + d)
    dout = torch.randn((q.shape[0], H, dv), generator=g).to(q.dtype)
    scale = default_scale(d)
    dq_, dk_, dv_, do_, cq, ck = (t.cuda() for t in (q, k, v, dout, cu_q, cu_k))
    mq, mk = max(lens_q + [0]), max(lens_k + [0])
    o, lse = fa.attention_forward_varlen(dq_, dk_, dv_, cq, ck, mq, causal=causal, scale=scale,
                                         dropout_p=p, seed=seed, offset=off)
    gq, gk, gv = fa.attention_backward_varlen(dq_, dk_, dv_, o, lse, do_, cq, ck, mq, mk,
                                              causal=causal, scale=scale, dropout_p=p, seed=seed,
                                              offset=off)
    torch.cuda.synchronize()
    assert fa.fa_status()[0] == fa.FA_OK
    o, lse, gq, gk, gv = (t.cpu() for t in (o, lse, gq, gk, gv))
    s = 256.0 / oracle.dropout_threshold(p)
    tmax, tmean = TOL[dtype]
    rq, rk, rv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    cq_l, ck_l = cu_q.tolist(), cu_k.tolist()
    for b in range(len(lens_q)):
        q0, q1, k0, k1 = cq_l[b], cq_l[b + 1], ck_l[b], ck_l[b + 1]
        shift = (k1 - k0) - (q1 - q0) if causal == "bottom_right" else 0
        for h in range(H):
            if q1 == q0:
                continue
            args = (q[q0:q1, h].double().numpy(), k[k0:k1, h].double().numpy(),
                    v[k0:k1, h].double().numpy())
            o_ref, l_ref = oracle.attention_dropout(*args, b * H + h, seed, off, p,
                                                    causal=causal is not None, scale=scale,
                                                    q_offset=shift)
            ob, lb = o[q0:q1, h].double().numpy(), lse[h, q0:q1].double().numpy()
            empty = np.isneginf(l_ref)
            assert np.all(np.isneginf(lb[empty])) and np.all(ob[empty] == 0.0)
            err = np.abs(ob[~empty] - o_ref[~empty])
            if err.size:
                assert err.max() <= tmax * s and err.mean() <= tmean * s, (name, b, h, err.max())
                assert np.abs(lb[~empty] - l_ref[~empty]).max() <= LSE_TOL
            if k1 > k0:
                gq_r, gk_r, gv_r = oracle.attention_dropout_grad(
                    *args, dout[q0:q1, h].double().numpy(), b * H + h, seed, off, p,
                    causal=causal is not None, scale=scale, q_offset=shift)
                rq[q0:q1, h], rk[k0:k1, h], rv[k0:k1, h] = gq_r, gk_r, gv_r
    check_grad(name + " dQ", gq, rq, dtype)
    check_grad(name + " dK", gk, rk, dtype)
    check_grad(name + " dV", gv, rv, dtype)


def test_kv_dropout_zero_probability_is_fa_fwd_kv():
    q, k, v = (t.cuda() for t in seeded_inputs.make_decode(2, 2, 200, 600, 64, "bf16", seed=5))
    o1, l1 = fa.attention_forward_kv(q, k, v, causal="bottom_right")
    o2, l2 = fa.attention_forward_kv(q, k, v, causal="bottom_right", dropout_p=0.0, seed=3, offset=1)
    lib = fa.load_library()
    o3 = torch.empty_like(o1)
    l3 = torch.empty_like(l1)
    assert fa.fa_fwd_kv_dropout(q, k, v, o3, l3, 2, 2, 200, 600, 64, 64, 2, None, 0.125, 0.0, 3, 1,
                                fa.FA_BF16) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(o1, o3) and torch.equal(l1, l3)
    assert lib is not None
