"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Small shapes cover every compiled variant (d 64/128 x bf16/fp16 x causal or
not) with ragged tails on both tile axes; the five synthetic workloads run at
full size in the same launch configuration the benchmark times, compared on
every row (small workloads) or on whole heads plus seeded random rows and
tile-edge rows (the long causal ones, where the float64 oracle cannot do
every row in seconds).
"""
import numpy as np
import pytest
import torch

import seeded_inputs
from gpu_common import (compare, default_scale, make, oracle_full, oracle_rows, require_gpu,
                        run_fa)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


SMALL = [
    # B, H, N, d, dtype, causal
    (1, 1, 1, 64, "bf16", False),
    (1, 1, 1, 128, "fp16", True),
    (1, 2, 7, 64, "fp16", True),
    (1, 1, 100, 128, "bf16", True),
    (1, 1, 128, 128, "bf16", False),
    (1, 1, 128, 64, "fp16", True),
    (2, 1, 129, 64, "bf16", False),
    (1, 2, 200, 128, "bf16", True),
    (2, 1, 256, 64, "fp16", False),
    (1, 1, 256, 128, "fp16", True),
    (1, 1, 300, 128, "fp16", False),
    (1, 3, 383, 64, "bf16", True),
    (1, 1, 384, 128, "bf16", False),
    (1, 1, 512, 128, "bf16", True),
    (2, 2, 640, 64, "fp16", True),
    (1, 2, 1000, 64, "fp16", False),
    (1, 1, 1111, 128, "bf16", False),
    (3, 1, 1500, 128, "fp16", True),
    (1, 2, 2049, 64, "bf16", True),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", SMALL,
                         ids=[f"B{c[0]}H{c[1]}N{c[2]}d{c[3]}{c[4]}{'c' if c[5] else ''}"
                              for c in SMALL])
def test_small_shapes_all_rows(B, H, N, d, dtype, causal):
    q, k, v = make(B, H, N, d, dtype, q_std=1.5, seed=N * 7 + d + causal)
    scale = default_scale(d)
    o, lse = run_fa(q, k, v, causal, scale)
    o_ref, lse_ref = oracle_full(q, k, v, causal, scale)
    compare(o, lse, o_ref, lse_ref, dtype, f"B{B}H{H}N{N}d{d}{dtype}")


@pytest.mark.parametrize("d,dtype,causal", [(64, "bf16", False), (128, "fp16", True)])
def test_other_scales(d, dtype, causal):
    q, k, v = make(1, 2, 333, d, dtype, seed=5)
    for scale in (0.02, 0.5):
        o, lse = run_fa(q, k, v, causal, scale)
        o_ref, lse_ref = oracle_full(q, k, v, causal, scale)
        compare(o, lse, o_ref, lse_ref, dtype, f"scale {scale}")


# ---------------------------------------------------------------- the five workloads

def _workload_inputs(name):
    w = seeded_inputs.workload(name)
    q, k, v = seeded_inputs.make_workload_qkv(w)
    return w, q, k, v


@pytest.mark.parametrize("name", ["b1_h1_n256_d64_fp16", "b16_h16_n1024_d64_bf16",
                                  "b1_h16_n4096_d128_bf16"])
def test_workload_every_row(name):
    w, q, k, v = _workload_inputs(name)
    o, lse = run_fa(q, k, v, w["causal"], w["scale"])
    o_ref, lse_ref = oracle_full(q, k, v, w["causal"], w["scale"])
    compare(o, lse, o_ref, lse_ref, w["dtype"], name)


def _sampled_rows(w, full_heads, count, seed):
    N = w["N"]
    edges = {0, 1, 127, 128, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1}
    sel = {}
    for bh in full_heads:
        sel[bh] = list(range(N))
    g = torch.Generator().manual_seed(seed)
    bs = torch.randint(0, w["B"], (count,), generator=g).tolist()
    hs = torch.randint(0, w["H"], (count,), generator=g).tolist()
    rs = torch.randint(0, N, (count,), generator=g).tolist()
    for b, h, r in zip(bs, hs, rs):
        sel.setdefault((b, h), set())
        if isinstance(sel[(b, h)], set):
            sel[(b, h)].add(r)
    last = (w["B"] - 1, w["H"] - 1)
    if not isinstance(sel.get(last), list):
        sel.setdefault(last, set()).update(edges)
    return {bh: sorted(set(rows)) for bh, rows in sel.items()}


@pytest.mark.parametrize("name,full_heads,count", [
    ("b4_h32_n8192_d128_bf16_causal", [(0, 0), (3, 31)], 4096),
    ("b1_h8_n32768_d64_fp16_causal_qstd4", [], 4096),
])
def test_workload_sampled_rows(name, full_heads, count):
    w, q, k, v = _workload_inputs(name)
    o, lse = run_fa(q, k, v, w["causal"], w["scale"])
    sel = _sampled_rows(w, full_heads, count, seed=w["seed"])
    if not full_heads:  # long context: the first 4096 rows of head 0 in full
        sel[(0, 0)] = sorted(set(sel.get((0, 0), [])) | set(range(4096)))
    ref = oracle_rows(q, k, v, w["causal"], w["scale"], sel)
    o_g = np.concatenate([o[b, h, rows].double().numpy() for (b, h), (rows, _, _) in ref.items()])
    l_g = np.concatenate([lse[b, h, rows].double().numpy() for (b, h), (rows, _, _) in ref.items()])
    o_r = np.concatenate([x[1] for x in ref.values()])
    l_r = np.concatenate([x[2] for x in ref.values()])
    compare(o_g, l_g, o_r, l_r, w["dtype"], name)
    # the rest of the output must at least be finite
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
