"""fa_decode (split-KV decoding) on the GPU against the float64 oracle.

Each query row is checked element by element against the oracle's exact
attention of that row over the cache, at its decoding position Nk - Nq + i
when causal.  Shapes cover one and several splits of the key axis, ragged
cache lengths, every supported query count edge (1 and 16), both head widths
and dtypes, an empty cache and causal queries placed before the cache.
Tolerances are the forward's (bf16 2e-2 / 2e-3, fp16 5e-3 / 5e-4 on O,
1e-3 on LSE).
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


def run_decode(q, k, v, causal, scale):
    o, lse = fa.attention_decode(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    return o.cpu(), lse.cpu()


def oracle_decode(q, k, v, causal, scale):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    pos = np.arange(Nq, dtype=np.int64) + (Nk - Nq)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = oracle.attention_rows(
                q[b, h].double().numpy(), pos, k[b, h].double().numpy().reshape(Nk, d),
                v[b, h].double().numpy().reshape(Nk, d), causal=causal, scale=scale)
    return o, lse


def check(o, lse, o_ref, lse_ref, dtype, what):
    o = o.double().numpy()
    lse = lse.double().numpy()
    assert np.all(np.isfinite(o)), what
    err = np.abs(o - o_ref)
    tmax, tmean = TOL[dtype]
    assert err.max() <= tmax and err.mean() <= tmean, f"{what}: O max {err.max():.3e} mean {err.mean():.3e}"
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf LSE rows differ"
    if (~empty).any():
        lerr = np.abs(lse[~empty] - lse_ref[~empty]).max()
        assert lerr <= LSE_TOL, f"{what}: LSE {lerr:.3e}"
    assert np.all(o[empty] == 0), f"{what}: empty rows must be zero"


SHAPES = [
    # B, H, Nq, Nk, d, dtype, causal
    (1, 1, 1, 1, 64, "fp16", False),
    (2, 3, 1, 100, 128, "bf16", False),
    (1, 4, 4, 1000, 64, "bf16", True),
    (2, 2, 16, 4097, 128, "fp16", True),
    (1, 8, 1, 65536, 128, "bf16", False),
    (3, 2, 5, 300, 64, "fp16", False),
    (1, 2, 16, 10, 128, "bf16", True),      # six queries sit before the cache: empty rows
    (1, 16, 2, 32768, 64, "fp16", True),
    (4, 8, 8, 3000, 128, "bf16", False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,causal", SHAPES,
                         ids=[f"B{s[0]}H{s[1]}q{s[2]}k{s[3]}d{s[4]}{s[5]}{'c' if s[6] else ''}" for s in SHAPES])
def test_decode_every_row(B, H, Nq, Nk, d, dtype, causal):
    seed = B * 131 + H * 17 + Nq * 7 + Nk + d
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, dtype, seed=seed)
    scale = default_scale(d)
    o, lse = run_decode(q, k, v, causal, scale)
    o_ref, lse_ref = oracle_decode(q, k, v, causal, scale)
    check(o, lse, o_ref, lse_ref, dtype, f"decode B{B} H{H} Nq{Nq} Nk{Nk} d{d}")


def test_decode_empty_cache():
    """Nk = 0: O = 0 and LSE = -inf (the pages' empty-key policy)."""
    q, _, _ = seeded_inputs.make_decode(2, 3, 4, 1, 64, "bf16", seed=1)
    k = torch.zeros(2, 3, 0, 64, dtype=torch.bfloat16)
    o, lse = run_decode(q, k, k, False, 0.125)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_decode_invariants():
    """V = ones gives O = 1; a second call gives identical bits."""
    q, k, v = seeded_inputs.make_decode(2, 4, 3, 5000, 128, "bf16", seed=2)
    ones = torch.ones_like(v)
    o, _ = run_decode(q, k, ones, True, 0.09)
    assert (o.double() - 1).abs().max().item() <= 1e-2
    a = run_decode(q, k, v, True, 0.09)
    b = run_decode(q, k, v, True, 0.09)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_matches_forward_last_rows():
    """Nq queries that are the last rows of a square causal problem give the
    same rows as fa_fwd (both against the same oracle, within tolerance)."""
    q, k, v = seeded_inputs.make_qkv(1, 4, 700, 64, "fp16", seed=3)
    o_f, l_f = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=True)
    o_d, l_d = fa.attention_decode(q[:, :, -8:].contiguous().cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert (o_f[:, :, -8:].double() - o_d.double()).abs().max().item() <= 2 * TOL["fp16"][0]
    assert (l_f[:, :, -8:] - l_d).abs().max().item() <= 2 * LSE_TOL


def test_decode_workspace_errors():
    q, k, v = (t.cuda() for t in seeded_inputs.make_decode(1, 2, 1, 5000, 64, "bf16", seed=4))
    need = fa.fa_decode_workspace_size(1, 2, 1, 5000, 64)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.attention_decode(q, k, v, workspace=small)
    assert e.value.code == fa.FA_ERR_WORKSPACE
