"""Properties of the CUDA path that hold at any size (through the C ABI).

These mirror the oracle's pins on the device: rows of softmax weights sum to
one, equal scores give the mean of V, N = 1 returns V, causal row 0 returns
V[0], the maximum arriving in the final key tile, a joint K/V permutation,
plus library properties: no writes outside O and LSE, determinism, no
memory allocated per call, stream ordering and the status word.
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
from gpu_common import TOL, compare, default_scale, make, oracle_full, require_gpu, run_fa

pytestmark = pytest.mark.gpu

VARIANTS = [(64, "bf16"), (64, "fp16"), (128, "bf16"), (128, "fp16")]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("d,dtype", VARIANTS)
@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(d, dtype, causal):
    q, k, _ = make(2, 2, 777, d, dtype, q_std=3.0, seed=1)
    v = torch.ones_like(q)
    o, _ = run_fa(q, k, v, causal)
    assert (o.double() - 1).abs().max().item() <= TOL[dtype][0]


@pytest.mark.parametrize("d,dtype", VARIANTS)
def test_equal_scores_give_mean(d, dtype):
    q, _, v = make(1, 2, 640, d, dtype, seed=2)
    k = torch.zeros_like(q)
    for causal in (False, True):
        o, lse = run_fa(q, k, v, causal)
        vd = v.double()
        if causal:
            cnt = torch.arange(1, 641, dtype=torch.float64)
            want = vd.cumsum(2) / cnt[:, None]
            want_lse = torch.log(cnt).expand(1, 2, 640)
        else:
            want = vd.mean(2, keepdim=True).expand_as(vd)
            want_lse = torch.full((1, 2, 640), math.log(640), dtype=torch.float64)
        compare(o, lse, want.numpy(), want_lse.numpy(), dtype, f"K=0 causal={causal}")


@pytest.mark.parametrize("d,dtype", VARIANTS)
def test_single_position_returns_v(d, dtype):
    q, k, v = make(3, 5, 1, d, dtype, seed=3)
    for causal in (False, True):
        o, lse = run_fa(q, k, v, causal)
        assert torch.equal(o, v)
        want = (q.double() * k.double()).sum(-1) * default_scale(d)
        assert (lse.double() - want).abs().max().item() <= 1e-3


@pytest.mark.parametrize("d,dtype", VARIANTS)
def test_causal_row0_returns_v0(d, dtype):
    q, k, v = make(2, 3, 500, d, dtype, q_std=4.0, seed=4)
    o, _ = run_fa(q, k, v, True)
    assert torch.equal(o[:, :, 0], v[:, :, 0])


@pytest.mark.parametrize("d,dtype", VARIANTS)
def test_maximum_in_final_key_tile(d, dtype):
    """Unremarkable keys, then one large score in the last tile: the rescale
    must pull all earlier tiles down (pages' late-maximum case, scaled up)."""
    N = 1000
    q, _, v = make(1, 1, N, d, dtype, seed=6)
    q = torch.zeros_like(q)
    q[..., 0] = 1.0
    k = torch.zeros_like(q)
    k[0, 0, N - 1, 0] = 30.0 * math.sqrt(d) / 2  # score 15 vs 0 elsewhere
    for causal in (False, True):
        o, lse = run_fa(q, k, v, causal)
        o_ref, lse_ref = oracle_full(q, k, v, causal, default_scale(d))
        compare(o, lse, o_ref, lse_ref, dtype, f"late max causal={causal}")


@pytest.mark.parametrize("d,dtype", VARIANTS)
def test_max_rises_every_tile(d, dtype):
    """Scores that grow key by key: every tile raises the maximum past the
    lazy-rescale threshold, so the O correction runs on every tile."""
    N = 1024
    q, _, v = make(1, 2, N, d, dtype, seed=7)
    q = torch.zeros_like(q)
    q[..., 0] = 1.0
    k = torch.zeros_like(q)
    ramp = torch.linspace(0, 60, N) * math.sqrt(d)   # scaled score rises to 60
    k[..., 0] = ramp.to(k.dtype)
    for causal in (False, True):
        o, lse = run_fa(q, k, v, causal)
        o_ref, lse_ref = oracle_full(q, k, v, causal, default_scale(d))
        compare(o, lse, o_ref, lse_ref, dtype, f"rising max causal={causal}")


@pytest.mark.parametrize("d,dtype", VARIANTS)
def test_joint_kv_permutation(d, dtype):
    q, k, v = make(1, 2, 900, d, dtype, seed=8)
    perm = torch.randperm(900, generator=torch.Generator().manual_seed(9))
    o1, l1 = run_fa(q, k, v, False)
    o2, l2 = run_fa(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False)
    assert (o1.double() - o2.double()).abs().max().item() <= TOL[dtype][0]
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_no_writes_outside_outputs():
    """Guard bands around O and LSE keep their sentinel (TMA stores clip at N)."""
    B, H, N, d = 1, 3, 300, 128
    q, k, v = (t.cuda() for t in make(B, H, N, d, "bf16", seed=10))
    n_o, n_l, pad = B * H * N * d, B * H * N, 4096
    o_buf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((n_l + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + n_o].view(B, H, N, d)
    lse = l_buf[pad:pad + n_l].view(B, H, N)
    for causal in (False, True):
        fa.attention_forward(q, k, v, causal=causal, out=o, lse=lse)
        torch.cuda.synchronize()
        assert (o_buf[:pad] == 7).all() and (o_buf[pad + n_o:] == 7).all()
        assert (l_buf[:pad] == 7).all() and (l_buf[pad + n_l:] == 7).all()
        assert torch.isfinite(o.float()).all()


def test_deterministic():
    q, k, v = (t.cuda() for t in make(2, 4, 1500, 64, "fp16", seed=11))
    a = fa.attention_forward(q, k, v, causal=True)
    b = fa.attention_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_no_device_memory_allocated_per_call():
    """The library allocates nothing: free device memory is unchanged by a
    long-sequence call whose N x N fp32 score matrix would need 4 GiB."""
    N = 32768
    q, k, v = (t.cuda() for t in make(1, 1, N, 64, "fp16", seed=12))
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, N, dtype=torch.float32, device="cuda")
    fa.attention_forward(q, k, v, causal=True, out=o, lse=lse)  # first call loads the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    fa.attention_forward(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free0 - free1) < (2 << 20)
    assert fa.fa_status()[0] == fa.FA_OK


def test_runs_on_a_side_stream():
    q, k, v = (t.cuda() for t in make(1, 2, 700, 128, "bf16", seed=13))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o, lse = fa.attention_forward(q, k, v, causal=True, stream=s)
    s.synchronize()
    o_ref, lse_ref = oracle_full(q.cpu(), k.cpu(), v.cpu(), True, default_scale(128))
    compare(o.cpu(), lse.cpu(), o_ref, lse_ref, "bf16", "side stream")


def test_empty_and_error_returns_on_device():
    q = torch.zeros(1, 1, 0, 64, dtype=torch.float16, device="cuda")
    o, lse = fa.attention_forward(q, q, q)
    assert o.shape == (1, 1, 0, 64) and lse.shape == (1, 1, 0)
    x = torch.zeros(1, 1, 64, 96, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.attention_forward(x, x, x)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED_D
    # 4 fp16 elements = 8 bytes past a 256-byte aligned allocation: not 16-byte aligned
    y = torch.zeros(1, 1, 64 * 64 + 4, dtype=torch.float16, device="cuda")[..., 4:].view(1, 1, 64, 64)
    with pytest.raises(fa.FaError) as e:
        fa.attention_forward(y, y, y)
    assert e.value.code == fa.FA_ERR_ALIGN
    assert fa.fa_status()[0] == fa.FA_OK
    _ = np
