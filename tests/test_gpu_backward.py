"""fa_bwd on the GPU against the float64 gradient oracle.

Inputs are the seeded Q, K, V of each shape, an independent seeded dO, and
the forward pass's own O and LSE (as a user's training step would pass
them).  The oracle differentiates the exact definition from the same
rounded Q, K, V and dO in float64.

Tolerance (derived from the arithmetic, stated relative to the largest
magnitude of each reference gradient): the kernels round P and dS to the
storage dtype before the tile GEMMs (relative error up to 2^-9 for bf16,
2^-12 for fp16), use the forward's 16-bit O for D = rowsum(dO * O), and
round the result once more; fp32 accumulation error is far below that.
Allowing about six rounding units at the largest magnitude for the worst
element and a tenth of that on average (a reference that is exactly zero,
as dQ and dK with a single key, is measured against magnitude 1e-3):
    bf16: max |err| <= 2.5e-2 * max|ref|, mean |err| <= 2.5e-3 * max|ref|
    fp16: max |err| <= 6e-3  * max|ref|, mean |err| <= 6e-4  * max|ref|
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import oracle
import seeded_inputs
from gpu_common import default_scale, make, require_gpu

pytestmark = pytest.mark.gpu

GRAD_TOL = {"bf16": (2.5e-2, 2.5e-3), "fp16": (6e-3, 6e-4)}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_bwd(q, k, v, dout, causal, scale):
    """Forward then backward on the GPU; returns CPU (dq, dk, dv)."""
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    o, lse = fa.attention_forward(dq_, dk_, dv_, causal=causal, scale=scale)
    gq, gk, gv = fa.attention_backward(dq_, dk_, dv_, o, lse, do_, causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    return gq.cpu(), gk.cpu(), gv.cpu()


def check_grad(name, gpu, ref, dtype):
    gpu = np.asarray(gpu.double() if torch.is_tensor(gpu) else gpu, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    # relative to the largest reference magnitude; an exactly-zero reference
    # (one key: dQ = dK = 0) is held to the same bound at magnitude 1e-3
    norm = max(float(np.abs(ref).max()), 1e-3)
    err = np.abs(gpu - ref)
    emax, emean = float(err.max()) / norm, float(err.mean()) / norm
    tmax, tmean = GRAD_TOL[dtype]
    assert emax <= tmax, f"{name}: max|err|/max|ref| {emax:.3e} > {tmax}"
    assert emean <= tmean, f"{name}: mean|err|/max|ref| {emean:.3e} > {tmean}"
    print(f"{name}: max {emax:.2e} mean {emean:.2e} (of max|ref| {norm:.3e})")
    return emax, emean


SHAPES = [
    # B, H, N, d, dtype, causal
    (1, 2, 1, 64, "bf16", False),
    (1, 2, 7, 128, "fp16", True),
    (1, 3, 100, 64, "bf16", False),
    (2, 2, 128, 128, "bf16", True),
    (1, 2, 129, 64, "fp16", True),
    (1, 2, 200, 128, "bf16", False),
    (2, 1, 256, 64, "bf16", True),
    (1, 2, 300, 128, "fp16", False),
    (1, 2, 383, 64, "fp16", True),
    (1, 1, 640, 128, "bf16", True),
    (1, 2, 1000, 64, "bf16", False),
    (1, 1, 1111, 128, "fp16", True),
    (1, 1, 1500, 64, "fp16", True),     # causal d = 64 past the 6-slot and 4-slot rings
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", SHAPES,
                         ids=[f"B{s[0]}H{s[1]}N{s[2]}d{s[3]}{s[4]}{'c' if s[5] else ''}" for s in SHAPES])
def test_backward_every_row(B, H, N, d, dtype, causal):
    seed = B * 7919 + H * 131 + N * 17 + d + int(causal)
    q, k, v = make(B, H, N, d, dtype, q_std=1.5, seed=seed)
    dout = seeded_inputs.make_dout(B, H, N, d, dtype, seed=seed)
    scale = default_scale(d)
    gq, gk, gv = run_bwd(q, k, v, dout, causal, scale)
    rq, rk, rv = oracle.attention_grad(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                       dout.double().numpy(), causal=causal, scale=scale)
    check_grad("dQ", gq, rq, dtype)
    check_grad("dK", gk, rk, dtype)
    check_grad("dV", gv, rv, dtype)


def test_backward_other_scale_and_large_scores():
    """A larger scale (peaked softmax, the forward's max moves often) stays exact."""
    q, k, v = make(1, 2, 384, 64, "fp16", q_std=3.0, seed=77)
    dout = seeded_inputs.make_dout(1, 2, 384, 64, "fp16", seed=77)
    for causal in (False, True):
        gq, gk, gv = run_bwd(q, k, v, dout, causal, 0.3)
        rq, rk, rv = oracle.attention_grad(q.double().numpy(), k.double().numpy(),
                                           v.double().numpy(), dout.double().numpy(),
                                           causal=causal, scale=0.3)
        check_grad("dQ", gq, rq, "fp16")
        check_grad("dK", gk, rk, "fp16")
        check_grad("dV", gv, rv, "fp16")


def test_backward_invariants():
    """sum_j dK_j = 0 per head; N = 1 gives dQ = dK = 0 and dV = dO; deterministic."""
    q, k, v = make(2, 2, 500, 128, "bf16", seed=5)
    dout = seeded_inputs.make_dout(2, 2, 500, 128, "bf16", seed=5)
    for causal in (False, True):
        gq, gk, gv = run_bwd(q, k, v, dout, causal, default_scale(128))
        ksum = gk.double().sum(dim=2).abs().max().item()
        assert ksum <= 2e-2 * gk.double().abs().max().item() * 500 ** 0.5
        gq2, gk2, gv2 = run_bwd(q, k, v, dout, causal, default_scale(128))
        assert torch.equal(gq, gq2) and torch.equal(gk, gk2) and torch.equal(gv, gv2)
    q1, k1, v1 = make(1, 4, 1, 64, "fp16", seed=6)
    d1 = seeded_inputs.make_dout(1, 4, 1, 64, "fp16", seed=6)
    gq, gk, gv = run_bwd(q1, k1, v1, d1, True, 0.125)
    assert gq.abs().max().item() <= 1e-3 and gk.abs().max().item() <= 1e-3
    assert (gv.double() - d1.double()).abs().max().item() <= 1e-3


@pytest.mark.parametrize("name", ["b1_h16_n4096_d128_bf16", "b16_h16_n1024_d64_bf16",
                                  "b4_h32_n8192_d128_bf16_causal",
                                  "b1_h8_n32768_d64_fp16_causal_qstd4"])
def test_backward_on_workloads(name):
    """Full-size workloads: two whole heads up to N = 4096, one beyond (dQ
    every row, dK and dV on sampled keys)."""
    w = seeded_inputs.workload(name)
    q, k, v = seeded_inputs.make_workload_qkv(w)
    dout = seeded_inputs.make_dout(w["B"], w["H"], w["N"], w["d"], w["dtype"], seed=w["seed"])
    gq, gk, gv = run_bwd(q, k, v, dout, w["causal"], w["scale"])
    N = w["N"]
    heads = [(0, 0), (w["B"] - 1, w["H"] - 1)] if N <= 4096 else [(0, 0)]
    keys = seeded_inputs.sample_rows(N, 192, seed=w["seed"],
                                     include=(0, 1, 127, 128, N // 2, N - 129, N - 128, N - 1))
    keys = np.asarray(keys, dtype=np.int64)
    for b, h in heads:
        qh, kh, vh, gh = (t[b, h].double().numpy() for t in (q, k, v, dout))
        rows = np.arange(N)
        rq, lse, delta = oracle.grad_query_rows(qh, gh, rows, kh, vh, causal=w["causal"],
                                                scale=w["scale"])
        rk, rv = oracle.grad_key_rows(kh[keys], vh[keys], keys, qh, gh, lse, delta,
                                      causal=w["causal"], scale=w["scale"])
        check_grad(f"{name} dQ head {b},{h}", gq[b, h], rq, w["dtype"])
        check_grad(f"{name} dK head {b},{h}", gk[b, h][keys], rk, w["dtype"])
        check_grad(f"{name} dV head {b},{h}", gv[b, h][keys], rv, w["dtype"])


def test_backward_errors():
    q = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 256, dtype=torch.float32, device="cuda")
    args = dict(q=q, k=q, v=q, o=q, lse=lse, dout=q, dq=q, dk=q, dv=q, delta=lse, B=1, H=1,
                N=256, d=64, causal=0, scale=0.125, dtype=fa.FA_BF16)
    assert fa.fa_bwd(**{**args, "d": 96}) == fa.FA_ERR_UNSUPPORTED_D
    assert fa.fa_bwd(**{**args, "delta": None}) == fa.FA_ERR_NULLPTR
    assert fa.fa_bwd(**{**args, "dk": q.data_ptr() + 8}) == fa.FA_ERR_ALIGN
    assert fa.fa_bwd(**{**args, "scale": 0.0}) == fa.FA_ERR_SCALE
    assert fa.fa_bwd(**{**args, "N": 0}) == fa.FA_OK
    assert fa.fa_bwd(**{**args, "B": -1}) == fa.FA_ERR_SHAPE
