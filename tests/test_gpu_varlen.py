"""fa_fwd_varlen (packed batches of sequences of different lengths) vs the
float64 oracle, through the C ABI.

Every sequence is handed to the oracle on its own: its query rows at their
absolute positions (row i at i for upper-left, at len_k - len_q + i for
bottom-right) against its own keys only, so a kernel that let one sequence
see another's keys, or wrote a row of one into another, fails.  Rows that
see no key must be exactly O = 0 and LSE = -inf.
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


def oracle_varlen(q, k, v, cu_q, cu_k, causal, scale):
    tq, H, _ = q.shape
    dv = v.shape[2]
    o = np.zeros((tq, H, dv))
    lse = np.zeros((H, tq))
    cq, ck = cu_q.tolist(), cu_k.tolist()
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 <= q0:
            continue
        pos = np.arange(q1 - q0, dtype=np.int64)
        if causal == "bottom_right":
            pos = pos + ((k1 - k0) - (q1 - q0))
        for h in range(H):
            ob, lb = oracle.attention_rows(q[q0:q1, h].double().numpy(), pos,
                                           k[k0:k1, h].double().numpy(),
                                           v[k0:k1, h].double().numpy(),
                                           causal=causal is not None, scale=scale)
            o[q0:q1, h], lse[h, q0:q1] = ob, lb
    return o, lse


def run_varlen(q, k, v, cu_q, cu_k, causal, scale, max_q=None):
    lens = (cu_q[1:] - cu_q[:-1]).tolist()
    max_q = max(lens + [0]) if max_q is None else max_q
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    o, lse = fa.attention_forward_varlen(dq, dk, dv, cu_q.cuda(), cu_k.cuda(), max_q,
                                         causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    return o.cpu(), lse.cpu()


def check(o, lse, o_ref, lse_ref, dtype, what):
    o = o.double().numpy()
    lse = lse.double().numpy()
    empty = np.isneginf(lse_ref)                      # [H, tq]
    assert np.all(np.isneginf(lse[empty])), f"{what}: empty rows must have LSE = -inf"
    assert np.all(o.transpose(1, 0, 2)[empty] == 0.0), f"{what}: empty rows must have O = 0"
    full = ~empty
    assert np.all(np.isfinite(lse[full])) and np.all(np.isfinite(o)), f"{what}: non-finite values"
    if not full.any():
        return
    err = np.abs(o - o_ref).transpose(1, 0, 2)[full]
    tmax, tmean = TOL[dtype]
    assert err.max() <= tmax, f"{what}: max|dO| {err.max():.3e}"
    assert err.mean() <= tmean, f"{what}: mean|dO| {err.mean():.3e}"
    lerr = np.abs(lse[full] - lse_ref[full]).max()
    assert lerr <= LSE_TOL, f"{what}: max|dLSE| {lerr:.3e}"


def seeded_lengths(n, lo, hi, seed):
    g = torch.Generator("cpu").manual_seed(600000 + seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


CASES = [
    # name, lens_q, lens_k, H, d, dv, dtype, causal
    ("edges_nc", [1, 127, 128, 129, 300, 0, 517], [1, 127, 128, 129, 300, 0, 517], 2, 64, 64,
     "bf16", None),
    ("edges_ul", [1, 127, 128, 129, 300, 0, 517], [1, 127, 128, 129, 300, 0, 517], 2, 128, 128,
     "fp16", "upper_left"),
    ("prefill_br", [64, 200, 1], [1000, 250, 3000], 2, 128, 64, "bf16", "bottom_right"),
    ("more_q_than_k", [300, 5, 40], [100, 0, 40], 1, 64, 128, "fp16", "bottom_right"),
    ("many_short", seeded_lengths(40, 1, 300, 1), seeded_lengths(40, 1, 300, 1), 3, 64, 64,
     "bf16", "upper_left"),
    ("cross_lengths", seeded_lengths(9, 1, 700, 2), seeded_lengths(9, 0, 900, 3), 2, 128, 128,
     "bf16", None),
]


@pytest.mark.parametrize("name,lens_q,lens_k,H,d,dv,dtype,causal", CASES, ids=[c[0] for c in CASES])
def test_varlen_vs_oracle(name, lens_q, lens_k, H, d, dv, dtype, causal):
    q, k, v, cu_q, cu_k = seeded_inputs.make_varlen(lens_q, lens_k, H, d, dtype,
                                                    seed=len(lens_q) + d + dv, dv=dv)
    scale = default_scale(d)
    o, lse = run_varlen(q, k, v, cu_q, cu_k, causal, scale)
    o_ref, lse_ref = oracle_varlen(q, k, v, cu_q, cu_k, causal, scale)
    check(o, lse, o_ref, lse_ref, dtype, name)


@pytest.mark.parametrize("d,dtype,causal", [(64, "bf16", "upper_left"), (128, "fp16", None),
                                            (128, "bf16", "bottom_right")])
def test_uniform_lengths_equal_fa_fwd_kv(d, dtype, causal):
    """Equal lengths packed token-major give bit-for-bit the output of
    fa_fwd_kv on the [B, H, N, d] layout: the same tiles, in the same order
    within each row, only addressed differently."""
    B, H, Nq, Nk = 3, 2, 333, 700
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, dtype, seed=41 + d)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    o1, l1 = fa.attention_forward_kv(dq, dk, dv, causal=causal)
    pq, pk, pv = (t.permute(0, 2, 1, 3).reshape(-1, H, d).contiguous() for t in (dq, dk, dv))
    cu_q = torch.arange(0, (B + 1) * Nq, Nq, dtype=torch.int32, device="cuda")
    cu_k = torch.arange(0, (B + 1) * Nk, Nk, dtype=torch.int32, device="cuda")
    o2, l2 = fa.attention_forward_varlen(pq, pk, pv, cu_q, cu_k, Nq, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o2.view(B, Nq, H, d).permute(0, 2, 1, 3), o1)
    assert torch.equal(l2.view(H, B, Nq).permute(1, 0, 2), l1)


def test_guard_bands_and_loose_max():
    """Writes stay inside O and LSE, and a max_seqlen_q above the longest
    sequence changes nothing."""
    lens_q, lens_k, H, d = [5, 260, 129], [300, 260, 1], 2, 128
    q, k, v, cu_q, cu_k = seeded_inputs.make_varlen(lens_q, lens_k, H, d, "bf16", seed=9)
    tq = q.shape[0]
    pad = 4096
    ob = torch.full((tq * H * d + 2 * pad,), 5.0, dtype=torch.bfloat16, device="cuda")
    lb = torch.full((H * tq + 2 * pad,), 5.0, dtype=torch.float32, device="cuda")
    o = ob[pad:pad + tq * H * d].view(tq, H, d)
    lse = lb[pad:pad + H * tq].view(H, tq)
    fa.attention_forward_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), 1000,
                                causal="bottom_right", out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(ob[:pad] == 5.0) and torch.all(ob[-pad:] == 5.0)
    assert torch.all(lb[:pad] == 5.0) and torch.all(lb[-pad:] == 5.0)
    o_ref, lse_ref = oracle_varlen(q, k, v, cu_q, cu_k, "bottom_right", default_scale(d))
    check(o.cpu(), lse.cpu(), o_ref, lse_ref, "bf16", "guard")


def test_offsets_out_of_range_are_clamped():
    """Offsets past the totals or decreasing ends are clamped by the kernel:
    nothing outside O and LSE is written and no error is raised."""
    H, d, tq, tk = 1, 64, 200, 300
    q, k, v, _, _ = seeded_inputs.make_varlen([tq], [tk], H, d, "fp16", seed=13)
    pad = 4096
    ob = torch.full((tq * H * d + 2 * pad,), 3.0, dtype=torch.float16, device="cuda")
    lb = torch.full((H * tq + 2 * pad,), 3.0, dtype=torch.float32, device="cuda")
    o = ob[pad:pad + tq * H * d].view(tq, H, d)
    lse = lb[pad:pad + H * tq].view(H, tq)
    cu_q = torch.tensor([0, 150, 100, 10 ** 6], dtype=torch.int32, device="cuda")
    cu_k = torch.tensor([-50, 300, 10 ** 6, 10 ** 7], dtype=torch.int32, device="cuda")
    fa.attention_forward_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q, cu_k, 300, causal=None,
                                out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_status()[0] == fa.FA_OK
    assert torch.all(ob[:pad] == 3.0) and torch.all(ob[-pad:] == 3.0)
    assert torch.all(lb[:pad] == 3.0) and torch.all(lb[-pad:] == 3.0)
    # sequence 2 is clamped to rows 100..199 (overlapping sequence 0, the
    # caller's error); rows 0..99 belong to sequence 0 alone: against keys
    # 0..299 (its start -50 clamped to 0)
    o_ref, lse_ref = oracle_varlen(q[:100], k, v, torch.tensor([0, 100]), torch.tensor([0, 300]),
                                   None, default_scale(d))
    check(o[:100].cpu(), lse[:, :100].cpu(), o_ref, lse_ref, "fp16", "clamped")


def test_empty_and_errors():
    q = torch.zeros(10, 1, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 10, dtype=torch.float32, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    z = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    s = 0.125
    # no keys at all: every row is empty
    assert fa.fa_fwd_varlen(q, None, None, o, lse, cu, z, 1, 1, 10, 10, 0, 64, 64, 2, s,
                            fa.FA_BF16) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    assert fa.fa_fwd_varlen(q, q, q, o, lse, cu, cu, 1, 1, 10, 10, 10, 64, 64, 3, s,
                            fa.FA_BF16) == fa.FA_ERR_SHAPE
    assert fa.fa_fwd_varlen(q, q, q, o, lse, None, cu, 1, 1, 10, 10, 10, 64, 64, 0, s,
                            fa.FA_BF16) == fa.FA_ERR_NULLPTR
    assert fa.fa_fwd_varlen(q, q, q, o, lse, cu.data_ptr() + 2, cu, 1, 1, 10, 10, 10, 64, 64, 0,
                            s, fa.FA_BF16) == fa.FA_ERR_ALIGN
    assert fa.fa_fwd_varlen(q, q, q, o, lse, cu, cu, 1, 1, 10, 10, 10, 64, 80, 0, s,
                            fa.FA_BF16) == fa.FA_ERR_UNSUPPORTED_D
    assert fa.fa_fwd_varlen(q, q, q, o, lse, cu, cu, 1, 1, 0, 10, 10, 64, 64, 0, s,
                            fa.FA_BF16) == fa.FA_OK
    assert fa.fa_status()[0] == fa.FA_OK
