"""fa_fwd_ws: the last round's units cut along the key axis and merged.

On a 152-SM GB300 the shapes below leave 4 to 118 units for the last
round, so the tail pieces range from single key tiles (more CTAs than tail
key tiles) to several tiles per piece, with ragged N and with units whose
second query tile lies past N.  Each result is compared with the float64
oracle (every row, or whole heads plus sampled rows) and with fa_fwd.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import seeded_inputs
from gpu_common import TOL, compare, default_scale, make, oracle_full, oracle_rows, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_ws(q, k, v, causal, scale, reuse=None):
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    ws = reuse if reuse is not None else fa.make_workspace(*q.shape, causal)
    o, lse = fa.attention_forward(dq, dk, dv, causal=causal, scale=scale, workspace=ws)
    o2, lse2 = fa.attention_forward(dq, dk, dv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    return o.cpu(), lse.cpu(), o2.cpu(), lse2.cpu(), ws


SHAPES = [
    # B, H, N, d, dtype
    (1, 40, 1024, 64, "bf16"),     # 160 units: 8 tail units, 64 tail key tiles < 152 CTAs
    (1, 39, 1000, 128, "bf16"),    # ragged N, 4 tail units
    (1, 80, 300, 64, "fp16"),      # second query tile of half the units lies past N
    (2, 45, 700, 128, "fp16"),     # 118 tail units, ~4.7 key tiles per CTA
    (3, 53, 520, 64, "bf16"),      # 3 key tiles per unit
]


@pytest.mark.parametrize("B,H,N,d,dtype", SHAPES, ids=[f"B{s[0]}H{s[1]}N{s[2]}d{s[3]}{s[4]}" for s in SHAPES])
def test_split_tail_every_row(B, H, N, d, dtype):
    q, k, v = make(B, H, N, d, dtype, q_std=2.0, seed=B * 1000 + H * 10 + N)
    scale = default_scale(d)
    o, lse, o_plain, lse_plain, ws = run_ws(q, k, v, False, scale)
    o_ref, lse_ref = oracle_full(q, k, v, False, scale)
    compare(o, lse, o_ref, lse_ref, dtype, "split")
    # same function as the unsplit kernel, up to rounding order
    assert (o.double() - o_plain.double()).abs().max().item() <= TOL[dtype][0]
    assert (lse - lse_plain).abs().max().item() <= 1e-3


@pytest.mark.parametrize("name", ["b1_h16_n4096_d128_bf16", "b16_h16_n1024_d64_bf16"])
def test_split_on_workloads(name):
    w = seeded_inputs.workload(name)
    q, k, v = seeded_inputs.make_workload_qkv(w)
    o, lse, o_plain, lse_plain, ws = run_ws(q, k, v, w["causal"], w["scale"])
    assert ws is not None, "these workloads leave a partial last round on 152 SMs"
    if w["B"] * w["H"] * w["N"] <= 65536:
        o_ref, lse_ref = oracle_full(q, k, v, False, w["scale"])
        compare(o, lse, o_ref, lse_ref, w["dtype"], name)
    else:
        sel = {(0, h): list(range(w["N"])) for h in (0, w["H"] - 1)}
        ref = oracle_rows(q, k, v, False, w["scale"], sel)
        o_g = np.concatenate([o[b, h, r].double().numpy() for (b, h), (r, _, _) in ref.items()])
        l_g = np.concatenate([lse[b, h, r].double().numpy() for (b, h), (r, _, _) in ref.items()])
        compare(o_g, l_g, np.concatenate([x[1] for x in ref.values()]),
                np.concatenate([x[2] for x in ref.values()]), w["dtype"], name)
    assert (o.double() - o_plain.double()).abs().max().item() <= TOL[w["dtype"]][0]


def test_workspace_reuse_is_deterministic():
    """Two calls sharing one workspace give identical results (counters reset)."""
    q, k, v = make(2, 45, 700, 128, "bf16", seed=31)
    o1, l1, _, _, ws = run_ws(q, k, v, False, default_scale(128))
    o2, l2, _, _, _ = run_ws(q, k, v, False, default_scale(128), reuse=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_workspace_size_and_errors():
    assert fa.fa_fwd_workspace_size(1, 40, 1024, 64, False) > 0
    assert fa.fa_fwd_workspace_size(1, 40, 1024, 64, True) == 0      # causal: never split
    assert fa.fa_fwd_workspace_size(1, 1, 256, 64, False) == 0       # one unit
    assert fa.fa_fwd_workspace_size(0, 4, 256, 64, False) == 0
    with pytest.raises(fa.FaError):
        fa.fa_fwd_workspace_size(1, 1, 256, 96, False)
    q, k, v = (t.cuda() for t in make(1, 40, 1024, 64, "bf16", seed=32))
    need = fa.fa_fwd_workspace_size(1, 40, 1024, 64, False)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.attention_forward(q, k, v, workspace=small)
    assert e.value.code == fa.FA_ERR_WORKSPACE
    # causal calls ignore the workspace and match fa_fwd exactly
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    a = fa.attention_forward(q, k, v, causal=True, workspace=ws)
    b = fa.attention_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert fa.fa_status()[0] == fa.FA_OK
