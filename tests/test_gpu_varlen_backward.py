"""fa_bwd_varlen (the backward pass of fa_fwd_varlen) vs the float64
gradient oracle, through the C ABI.

Every sequence goes to the oracle on its own: dQ (with its LSE and D) at
each query's absolute position against the sequence's keys, then dK, dV of
those keys with positions shifted by the query offset, so gradients that
leaked between sequences or rows written into a neighbour fail.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import oracle
import seeded_inputs
from gpu_common import default_scale, require_gpu
from test_gpu_backward import check_grad
from test_gpu_varlen import seeded_lengths

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def oracle_varlen_grad(q, k, v, dout, cu_q, cu_k, causal, scale):
    gq, gk, gv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    cq, ck = cu_q.tolist(), cu_k.tolist()
    H = q.shape[1]
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        nq, n = q1 - q0, k1 - k0
        off = n - nq if causal == "bottom_right" else 0
        pos = np.arange(nq, dtype=np.int64) + off
        for h in range(H):
            qh, gh = q[q0:q1, h].double().numpy(), dout[q0:q1, h].double().numpy()
            kh, vh = k[k0:k1, h].double().numpy(), v[k0:k1, h].double().numpy()
            if nq:
                dq, lse, delta = oracle.grad_query_rows(qh, gh, pos, kh, vh,
                                                        causal=causal is not None, scale=scale)
                gq[q0:q1, h] = dq
            if n and nq:
                dk, dv = oracle.grad_key_rows(kh, vh, np.arange(n, dtype=np.int64) - off, qh, gh,
                                              lse, delta, causal=causal is not None, scale=scale)
                gk[k0:k1, h], gv[k0:k1, h] = dk, dv
    return gq, gk, gv


CASES = [
    # name, lens_q, lens_k, H, d, dtype, causal
    ("edges_ul", [1, 127, 129, 300, 0, 517], [1, 127, 129, 300, 0, 517], 2, 64, "bf16",
     "upper_left"),
    ("prefill_br", [64, 200, 1], [1000, 250, 3000], 2, 128, "fp16", "bottom_right"),
    ("more_q_than_k", [300, 5, 40], [100, 0, 40], 1, 64, "fp16", "bottom_right"),
    ("cross_nc", seeded_lengths(9, 1, 700, 2), seeded_lengths(9, 1, 900, 3), 2, 128, "bf16", None),
    ("many_short", seeded_lengths(30, 1, 200, 1), seeded_lengths(30, 1, 200, 1), 2, 64, "bf16",
     "upper_left"),
]


@pytest.mark.parametrize("name,lens_q,lens_k,H,d,dtype,causal", CASES, ids=[c[0] for c in CASES])
def test_varlen_backward_vs_oracle(name, lens_q, lens_k, H, d, dtype, causal):
    q, k, v, cu_q, cu_k = seeded_inputs.make_varlen(lens_q, lens_k, H, d, dtype,
                                                    seed=len(lens_q) + 7 * d)
    g = torch.Generator("cpu").manual_seed(len(lens_q))
    dout = torch.randn(q.shape, generator=g).to(q.dtype)
    scale = default_scale(d)
    dq_, dk_, dv_, do_, cq, ck = (t.cuda() for t in (q, k, v, dout, cu_q, cu_k))
    mq, mk = max(lens_q + [0]), max(lens_k + [0])
    o, lse = fa.attention_forward_varlen(dq_, dk_, dv_, cq, ck, mq, causal=causal, scale=scale)
    gq, gk, gv = fa.attention_backward_varlen(dq_, dk_, dv_, o, lse, do_, cq, ck, mq, mk,
                                              causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    rq, rk, rv = oracle_varlen_grad(q, k, v, dout, cu_q, cu_k, causal, scale)
    check_grad(name + " dQ", gq.cpu(), rq, dtype)
    check_grad(name + " dK", gk.cpu(), rk, dtype)
    check_grad(name + " dV", gv.cpu(), rv, dtype)


WIDTH_CASES = [
    # name, lens_q, lens_k, H, d, dv, dtype, causal
    ("qk64_v128_ul", [1, 127, 129, 300, 0, 517], [1, 127, 129, 300, 0, 517], 2, 64, 128, "bf16",
     "upper_left"),
    ("qk128_v64_br", [64, 200, 1], [1000, 250, 3000], 2, 128, 64, "fp16", "bottom_right"),
]


@pytest.mark.parametrize("name,lens_q,lens_k,H,d,dv,dtype,causal", WIDTH_CASES,
                         ids=[c[0] for c in WIDTH_CASES])
def test_varlen_backward_value_width(name, lens_q, lens_k, H, d, dv, dtype, causal):
    """Values (and O, dO, dV) of another width than queries and keys."""
    q, k, v, cu_q, cu_k = seeded_inputs.make_varlen(lens_q, lens_k, H, d, dtype,
                                                    seed=len(lens_q) + 7 * d + dv, dv=dv)
    g = torch.Generator("cpu").manual_seed(len(lens_q) + dv)
    dout = torch.randn((q.shape[0], H, dv), generator=g).to(q.dtype)
    scale = default_scale(d)
    dq_, dk_, dv_, do_, cq, ck = (t.cuda() for t in (q, k, v, dout, cu_q, cu_k))
    mq, mk = max(lens_q + [0]), max(lens_k + [0])
    o, lse = fa.attention_forward_varlen(dq_, dk_, dv_, cq, ck, mq, causal=causal, scale=scale)
    gq, gk, gv = fa.attention_backward_varlen(dq_, dk_, dv_, o, lse, do_, cq, ck, mq, mk,
                                              causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    assert gq.shape == q.shape and gk.shape == k.shape and gv.shape == v.shape
    rq, rk, rv = oracle_varlen_grad(q, k, v, dout, cu_q, cu_k, causal, scale)
    check_grad(name + " dQ", gq.cpu(), rq, dtype)
    check_grad(name + " dK", gk.cpu(), rk, dtype)
    check_grad(name + " dV", gv.cpu(), rv, dtype)


@pytest.mark.parametrize("d,dtype,causal", [(64, "bf16", "upper_left"), (128, "fp16", None),
                                            (128, "bf16", "bottom_right")])
def test_uniform_lengths_equal_fa_bwd_kv(d, dtype, causal):
    """Equal lengths packed token-major: bit for bit the gradients of
    fa_bwd_kv on the [B, H, N, d] layout."""
    B, H, Nq, Nk = 3, 2, 333, 700
    q, k, v = (t.cuda() for t in seeded_inputs.make_decode(B, H, Nq, Nk, d, dtype, seed=43 + d))
    do = seeded_inputs.make_dout(B, H, Nq, d, dtype, seed=43).cuda()
    o1, l1 = fa.attention_forward_kv(q, k, v, causal=causal)
    g1 = fa.attention_backward_kv(q, k, v, o1, l1, do, causal=causal)
    pack = lambda t: t.permute(0, 2, 1, 3).reshape(-1, H, d).contiguous()   # noqa: E731
    cu_q = torch.arange(0, (B + 1) * Nq, Nq, dtype=torch.int32, device="cuda")
    cu_k = torch.arange(0, (B + 1) * Nk, Nk, dtype=torch.int32, device="cuda")
    pq, pk, pv, pdo = pack(q), pack(k), pack(v), pack(do)
    o2, l2 = fa.attention_forward_varlen(pq, pk, pv, cu_q, cu_k, Nq, causal=causal)
    g2 = fa.attention_backward_varlen(pq, pk, pv, o2, l2, pdo, cu_q, cu_k, Nq, Nk, causal=causal)
    torch.cuda.synchronize()
    for a, b, n in zip(g1, g2, (Nq, Nk, Nk)):
        assert torch.equal(b.view(B, n, H, d).permute(0, 2, 1, 3), a)


def test_varlen_backward_guard_bands():
    """Gradient writes stay inside dQ, dK and dV (a sequence past the others
    and a loose max_seqlen)."""
    lens_q, lens_k, H, d = [5, 260, 129], [300, 260, 1], 2, 64
    q, k, v, cu_q, cu_k = seeded_inputs.make_varlen(lens_q, lens_k, H, d, "bf16", seed=12)
    dout = torch.randn(q.shape, generator=torch.Generator("cpu").manual_seed(3)).to(q.dtype)
    dq_, dk_, dv_, do_, cq, ck = (t.cuda() for t in (q, k, v, dout, cu_q, cu_k))
    o, lse = fa.attention_forward_varlen(dq_, dk_, dv_, cq, ck, 600, causal="bottom_right")
    pad = 4096
    outs = []
    for shape in (q.shape, k.shape, v.shape):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), 9.0, dtype=q.dtype, device="cuda")
        outs.append((buf, buf[pad:pad + n].view(shape)))
    delta = torch.empty((q.shape[0], H), dtype=torch.float32, device="cuda")
    rc = fa.fa_bwd_varlen(dq_, dk_, dv_, o, lse, do_, outs[0][1], outs[1][1], outs[2][1], delta, cq,
                          ck, 3, H, 600, 700, q.shape[0], k.shape[0], d, d, 2, default_scale(d),
                          fa.FA_BF16)
    torch.cuda.synchronize()
    assert rc == fa.FA_OK and fa.fa_status()[0] == fa.FA_OK
    for buf, _ in outs:
        assert torch.all(buf[:pad] == 9.0) and torch.all(buf[-pad:] == 9.0)
    rq, rk, rv = oracle_varlen_grad(q, k, v, dout, cu_q, cu_k, "bottom_right", default_scale(d))
    check_grad("guard dQ", outs[0][1].cpu(), rq, "bf16")
    check_grad("guard dK", outs[1][1].cpu(), rk, "bf16")
    check_grad("guard dV", outs[2][1].cpu(), rv, "bf16")
