"""fa_bwd_onepass and fa_bwd_onepass_dropout on the GPU: the float64
gradient oracles, and fa_bwd / fa_bwd_dropout.

The one-pass kernel visits each (query tile, key tile) pair once and sums
dQ in fp32 through a workspace (the fp32 additions of different key tiles
arrive in no fixed order).  Its dK and dV come from the same tile products
on the same 16-bit operands as fa_bwd's, so they must equal fa_bwd's bit
for bit; dQ is held to the gradient tolerance of tests/test_gpu_backward.py
against the oracle.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import oracle
import seeded_inputs
from gpu_common import default_scale, make, require_gpu
from test_gpu_backward import SHAPES, check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def status_ok():
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"


def run_both(q, k, v, dout, causal, scale):
    """Forward, then fa_bwd and fa_bwd_onepass on the same O and LSE."""
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    o, lse = fa.attention_forward(dq_, dk_, dv_, causal=causal, scale=scale)
    two = fa.attention_backward(dq_, dk_, dv_, o, lse, do_, causal=causal, scale=scale)
    one = fa.attention_backward_onepass(dq_, dk_, dv_, o, lse, do_, causal=causal, scale=scale)
    status_ok()
    return [t.cpu() for t in two], [t.cpu() for t in one]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", SHAPES,
                         ids=[f"B{s[0]}H{s[1]}N{s[2]}d{s[3]}{s[4]}{'c' if s[5] else ''}" for s in SHAPES])
def test_onepass_every_row(B, H, N, d, dtype, causal):
    seed = B * 7919 + H * 131 + N * 17 + d + int(causal)
    q, k, v = make(B, H, N, d, dtype, q_std=1.5, seed=seed)
    dout = seeded_inputs.make_dout(B, H, N, d, dtype, seed=seed)
    scale = default_scale(d)
    (_, tk, tv), (gq, gk, gv) = run_both(q, k, v, dout, causal, scale)
    rq, rk, rv = oracle.attention_grad(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                       dout.double().numpy(), causal=causal, scale=scale)
    check_grad("dQ", gq, rq, dtype)
    check_grad("dK", gk, rk, dtype)
    check_grad("dV", gv, rv, dtype)
    assert torch.equal(gk, tk), "dK differs from fa_bwd"
    assert torch.equal(gv, tv), "dV differs from fa_bwd"


@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "fp16")])
def test_partial_head_group(d, dtype):
    """Causal calls deal work items in groups of 8 heads; with B*H = 12 the
    last group holds 4.  Both backward paths against the oracle."""
    B, H, N = 3, 4, 300
    q, k, v = make(B, H, N, d, dtype, q_std=1.5, seed=31 + d)
    dout = seeded_inputs.make_dout(B, H, N, d, dtype, seed=31 + d)
    scale = default_scale(d)
    (tq, tk, tv), (gq, gk, gv) = run_both(q, k, v, dout, True, scale)
    rq, rk, rv = oracle.attention_grad(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                       dout.double().numpy(), causal=True, scale=scale)
    for name, (a, b, c) in (("fa_bwd", (tq, tk, tv)), ("fa_bwd_onepass", (gq, gk, gv))):
        check_grad(f"{name} dQ", a, rq, dtype)
        check_grad(f"{name} dK", b, rk, dtype)
        check_grad(f"{name} dV", c, rv, dtype)


def test_onepass_repeat_and_workspace_reuse():
    """A reused (dirty) workspace gives the same dK, dV and a dQ within
    fp32 summation-order noise; a larger workspace than needed is fine."""
    q, k, v = make(2, 2, 700, 64, "bf16", seed=11)
    dout = seeded_inputs.make_dout(2, 2, 700, 64, "bf16", seed=11)
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    o, lse = fa.attention_forward(dq_, dk_, dv_, causal=True)
    need = fa.fa_bwd_onepass_workspace_size(2, 2, 700, 64)
    assert need == 2 * 2 * 64 * 768 * 4
    ws = torch.full((need + 4096,), 0x7F, dtype=torch.uint8, device="cuda")
    a = fa.attention_backward_onepass(dq_, dk_, dv_, o, lse, do_, causal=True, workspace=ws)
    b = fa.attention_backward_onepass(dq_, dk_, dv_, o, lse, do_, causal=True, workspace=ws)
    status_ok()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    diff = (a[0].double() - b[0].double()).abs().max().item()
    assert diff <= 2 ** -7 * a[0].double().abs().max().item()


@pytest.mark.parametrize("name", ["b1_h16_n4096_d128_bf16", "b1_h8_n32768_d64_fp16_causal_qstd4"])
def test_onepass_on_workloads(name):
    """Full-size workloads on the persistent grid: dQ of a whole head against
    the oracle (and of the last head for N <= 4096), dK and dV equal to
    fa_bwd's everywhere and checked on sampled keys."""
    w = seeded_inputs.workload(name)
    q, k, v = seeded_inputs.make_workload_qkv(w)
    dout = seeded_inputs.make_dout(w["B"], w["H"], w["N"], w["d"], w["dtype"], seed=w["seed"])
    (_, tk, tv), (gq, gk, gv) = run_both(q, k, v, dout, w["causal"], w["scale"])
    assert torch.equal(gk, tk) and torch.equal(gv, tv)
    N = w["N"]
    heads = [(0, 0), (w["B"] - 1, w["H"] - 1)] if N <= 4096 else [(0, 0)]
    keys = seeded_inputs.sample_rows(N, 96, seed=w["seed"],
                                     include=(0, 1, 127, 128, N // 2, N - 129, N - 128, N - 1))
    keys = np.asarray(keys, dtype=np.int64)
    for b, h in heads:
        qh, kh, vh, gh = (t[b, h].double().numpy() for t in (q, k, v, dout))
        rq, lse, delta = oracle.grad_query_rows(qh, gh, np.arange(N), kh, vh, causal=w["causal"],
                                                scale=w["scale"])
        rk, rv = oracle.grad_key_rows(kh[keys], vh[keys], keys, qh, gh, lse, delta,
                                      causal=w["causal"], scale=w["scale"])
        check_grad(f"{name} dQ head {b},{h}", gq[b, h], rq, w["dtype"])
        check_grad(f"{name} dK head {b},{h}", gk[b, h][keys], rk, w["dtype"])
        check_grad(f"{name} dV head {b},{h}", gv[b, h][keys], rv, w["dtype"])


DROP_CASES = [
    # B, H, N, d, dtype, causal, p, seed, offset: the dropout backward cases
    # of tests/test_gpu_dropout.py, a causal d = 128 shape past one ring
    # cycle, and an unmasked d = 64 shape with several tiles
    (1, 2, 300, 64, "bf16", True, 0.1, 1234, 0),
    (2, 1, 257, 128, "fp16", False, 0.5, 7, 3),
    (1, 1, 129, 128, "bf16", True, 0.3, 2 ** 40 + 3, 11),
    (1, 2, 640, 64, "fp16", False, 0.2, 99, 2 ** 31 + 5),
    (1, 1, 1000, 128, "bf16", True, 0.1, 5, 6),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,p,seed,off", DROP_CASES,
                         ids=[f"B{c[0]}H{c[1]}N{c[2]}d{c[3]}{c[4]}{'c' if c[5] else ''}p{c[6]}"
                              for c in DROP_CASES])
def test_onepass_dropout_vs_oracle(B, H, N, d, dtype, causal, p, seed, off):
    """fa_bwd_onepass_dropout against the float64 dropout gradient oracle;
    dK and dV equal fa_bwd_dropout's bit for bit."""
    q, k, v = seeded_inputs.make_qkv(B, H, N, d, dtype, 1.0, seed=N + d)
    dout = seeded_inputs.make_dout(B, H, N, d, dtype, seed=N + d)
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    o, lse = fa.attention_forward_dropout(dq_, dk_, dv_, p, seed, off, causal=causal)
    _, tk, tv = fa.attention_backward_dropout(dq_, dk_, dv_, o, lse, do_, p, seed, off,
                                              causal=causal)
    gq, gk, gv = fa.attention_backward_onepass(dq_, dk_, dv_, o, lse, do_, causal=causal,
                                               dropout_p=p, seed=seed, offset=off)
    status_ok()
    scale = default_scale(d)
    name = f"B{B}H{H}N{N}d{d}{dtype} p={p}"
    for b in range(B):
        for h in range(H):
            rq, rk, rv = oracle.attention_dropout_grad(
                q[b, h].double().numpy(), k[b, h].double().numpy(), v[b, h].double().numpy(),
                dout[b, h].double().numpy(), b * H + h, seed, off, p, causal=causal, scale=scale)
            check_grad(f"{name} ({b},{h}) dQ", gq[b, h].cpu(), rq, dtype)
            check_grad(f"{name} ({b},{h}) dK", gk[b, h].cpu(), rk, dtype)
            check_grad(f"{name} ({b},{h}) dV", gv[b, h].cpu(), rv, dtype)
    assert torch.equal(gk, tk), "dK differs from fa_bwd_dropout"
    assert torch.equal(gv, tv), "dV differs from fa_bwd_dropout"


def test_onepass_dropout_zero_probability_and_errors():
    """p = 0 gives fa_bwd_onepass's dK and dV; a bad probability is refused
    before the other checks."""
    q, k, v = (t.cuda() for t in make(1, 2, 300, 64, "bf16", seed=8))
    dout = seeded_inputs.make_dout(1, 2, 300, 64, "bf16", seed=8).cuda()
    o, lse = fa.attention_forward(q, k, v, causal=True)
    a = fa.attention_backward_onepass(q, k, v, o, lse, dout, causal=True)
    need = fa.fa_bwd_onepass_workspace_size(1, 2, 300, 64)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty(1, 2, 300, dtype=torch.float32, device="cuda")
    args = (q, k, v, o, lse, dout, dq, dk, dv, delta, 1, 2, 300, 64, 1, 0.125)
    assert fa.fa_bwd_onepass_dropout(*args, 0.0, 1, 2, fa.FA_BF16, ws, need) == fa.FA_OK
    status_ok()
    assert torch.equal(dk, a[1]) and torch.equal(dv, a[2])
    assert fa.fa_bwd_onepass_dropout(*args, 1.0, 1, 2, fa.FA_BF16, ws, need) == fa.FA_ERR_DROPOUT
    assert fa.fa_bwd_onepass_dropout(*args, 0.1, 1, 2, fa.FA_BF16, None, 0) == fa.FA_ERR_WORKSPACE


def test_onepass_errors():
    q = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 256, dtype=torch.float32, device="cuda")
    need = fa.fa_bwd_onepass_workspace_size(1, 1, 256, 64)
    ws = torch.zeros(need + 16, dtype=torch.uint8, device="cuda")
    args = dict(q=q, k=q, v=q, o=q, lse=lse, dout=q, dq=q, dk=q, dv=q, delta=lse, B=1, H=1,
                N=256, d=64, causal=0, scale=0.125, dtype=fa.FA_BF16, workspace=ws,
                workspace_bytes=need)
    assert fa.fa_bwd_onepass(**{**args, "workspace": None}) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd_onepass(**{**args, "workspace_bytes": need - 4}) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd_onepass(**{**args, "workspace": ws.data_ptr() + 8}) == fa.FA_ERR_ALIGN
    assert fa.fa_bwd_onepass(**{**args, "d": 96}) == fa.FA_ERR_UNSUPPORTED_D
    assert fa.fa_bwd_onepass(**{**args, "N": 0}) == fa.FA_OK
    assert fa.fa_bwd_onepass(**args) == fa.FA_OK
    status_ok()
