"""Helpers shared by the GPU tests: running the CUDA path and comparing with the oracle."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import oracle
import seeded_inputs

# Tolerances on O (max and mean |dO|) per storage dtype, and on LSE (absolute).
TOL = {"bf16": (2e-2, 2e-3), "fp16": (5e-3, 5e-4)}
LSE_TOL = 1e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    fa.load_library()  # raises when the CUDA library is missing


def run_fa(q, k, v, causal, scale=None, stream=None):
    """CUDA path on device copies of CPU tensors q, k, v; returns CPU (o, lse)."""
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    o, lse = fa.attention_forward(dq, dk, dv, causal=causal, scale=scale, stream=stream)
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"
    return o.cpu(), lse.cpu()


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    """Element-wise check against the oracle; returns (max, mean, lse max) errors."""
    o_gpu = np.asarray(o_gpu.double() if torch.is_tensor(o_gpu) else o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu.double() if torch.is_tensor(lse_gpu) else lse_gpu,
                         dtype=np.float64)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse_gpu)), f"{what}: non-finite LSE"
    err = np.abs(o_gpu - o_ref)
    emax, emean = float(err.max()), float(err.mean())
    lmax = float(np.abs(lse_gpu - lse_ref).max())
    tmax, tmean = TOL[dtype]
    assert emax <= tmax, f"{what}: max|dO| {emax:.3e} > {tmax}"
    assert emean <= tmean, f"{what}: mean|dO| {emean:.3e} > {tmean}"
    assert lmax <= LSE_TOL, f"{what}: max|dLSE| {lmax:.3e} > {LSE_TOL}"
    return emax, emean, lmax


def oracle_full(q, k, v, causal, scale):
    o, lse = oracle.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                              causal=causal, scale=scale)
    return o, lse


def oracle_rows(q, k, v, causal, scale, bh_rows):
    """Oracle on selected rows: bh_rows = {(b, h): [rows]} -> {(b, h): (rows, o, lse)}."""
    out = {}
    for (b, h), rows in bh_rows.items():
        rows = np.asarray(sorted(rows), dtype=np.int64)
        qr = q[b, h, rows].double().numpy()
        o, lse = oracle.attention_rows(qr, rows, k[b, h].double().numpy(),
                                       v[b, h].double().numpy(), causal=causal, scale=scale)
        out[(b, h)] = (rows, o, lse)
    return out


def default_scale(d):
    return 1.0 / math.sqrt(d)


def make(B, H, N, d, dtype, q_std=1.0, seed=0):
    return seeded_inputs.make_qkv(B, H, N, d, dtype, q_std, seed)
