"""Seeded synthetic inputs for the attention workloads.

This module is shared by the CUDA path's tests and benchmark and by the
float64 oracle's tests.  It holds no attention arithmetic: it only draws
random numbers, rounds them to the storage dtype, and names the workloads.

Recipe (the pages fix no generator): ``torch.Generator('cpu')`` seeded with
the workload's seed; Q, then K, then V, each drawn as float32 ``randn`` of
shape [B, H, N, d]; Q multiplied by ``q_std``; all three rounded to the
workload dtype (round-to-nearest-even, torch's ``.to``).  Both sides of a
parity test see exactly these rounded values (the oracle upcasts them to
float64).
"""
import itertools
import math

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}

# The five synthetic workloads: shape, storage dtype, mask and Q spread.  All
# use scale = 1/sqrt(d).  Seeds are 1000 + position in this list.
WORKLOADS = [
    dict(name="b1_h1_n256_d64_fp16", B=1, H=1, N=256, d=64, dtype="fp16",
         causal=False, q_std=1.0),
    dict(name="b1_h16_n4096_d128_bf16", B=1, H=16, N=4096, d=128, dtype="bf16",
         causal=False, q_std=1.0),
    dict(name="b4_h32_n8192_d128_bf16_causal", B=4, H=32, N=8192, d=128,
         dtype="bf16", causal=True, q_std=1.0),
    dict(name="b1_h8_n32768_d64_fp16_causal_qstd4", B=1, H=8, N=32768, d=64,
         dtype="fp16", causal=True, q_std=4.0),
    dict(name="b16_h16_n1024_d64_bf16", B=16, H=16, N=1024, d=64, dtype="bf16",
         causal=False, q_std=1.0),
]
for _i, _w in enumerate(WORKLOADS):
    _w["seed"] = 1000 + _i
    _w["scale"] = 1.0 / math.sqrt(_w["d"])


# Decoding workloads (split-KV, fa_decode): Nq new queries per head against a
# cache of Nk keys.  The pages print no decoding configuration; these take
# the causal long-context workload's cache (B1 H8 N32768 d64 fp16) and a
# larger batch of heads at d128, one new query each, causal.  Seeds 2000 + i.
DECODE_WORKLOADS = [
    dict(name="decode_b1_h8_q1_k32768_d64_fp16", B=1, H=8, Nq=1, Nk=32768, d=64, dtype="fp16",
         causal=True),
    dict(name="decode_b8_h32_q1_k32768_d128_bf16", B=8, H=32, Nq=1, Nk=32768, d=128,
         dtype="bf16", causal=True),
]
for _i, _w in enumerate(DECODE_WORKLOADS):
    _w["seed"] = 2000 + _i
    _w["scale"] = 1.0 / math.sqrt(_w["d"])


# Queries against a key set of another length (fa_fwd_kv).  The pages name
# chunked prefill after a cache and padded batches but print no sizes; these
# are: a 2048-query chunk appended to a 14336-key cache (bottom-right causal,
# B4 H32 d128 bf16), and a padded batch of 16 with per-batch key counts drawn
# uniformly from [Nk/8, Nk] (unmasked, B16 H16 Nq1024 Nk2048 d64 bf16).
# Seeds 3000 + i; key counts from ``make_seqlens``.
KV_WORKLOADS = [
    dict(name="prefill_b4_h32_q2048_k16384_d128_bf16_bottom_right", B=4, H=32, Nq=2048,
         Nk=16384, d=128, dtype="bf16", causal="bottom_right", padded=False),
    dict(name="padded_b16_h16_q1024_k2048_d64_bf16", B=16, H=16, Nq=1024, Nk=2048, d=64,
         dtype="bf16", causal=None, padded=True),
]
for _i, _w in enumerate(KV_WORKLOADS):
    _w["seed"] = 3000 + _i
    _w["scale"] = 1.0 / math.sqrt(_w["d"])


# Packed variable-length batches (fa_fwd_varlen): self-attention over B
# sequences whose lengths are uniform integers in [lo, hi] (seeded), query
# and key lengths equal, upper-left causal (a prefill of mixed prompts).
# The pages give no sizes; seed 4000 + i.
VARLEN_WORKLOADS = [
    dict(name="varlen_b16_h16_len256to4096_d128_bf16_causal", B=16, H=16, d=128, dtype="bf16",
         causal="upper_left", lo=256, hi=4096),
]
for _i, _w in enumerate(VARLEN_WORKLOADS):
    _w["seed"] = 4000 + _i
    _w["scale"] = 1.0 / math.sqrt(_w["d"])


def varlen_workload(name):
    """The fa_fwd_varlen workload dict with this name."""
    for w in VARLEN_WORKLOADS:
        if w["name"] == name:
            return dict(w)
    raise KeyError(name)


def varlen_lengths(B, lo, hi, seed):
    """Sequence lengths, uniform integers in [lo, hi], from their own
    generator (seeded 610000 + seed)."""
    g = torch.Generator("cpu").manual_seed(610000 + int(seed))
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


def kv_workload(name):
    """The fa_fwd_kv workload dict with this name."""
    for w in KV_WORKLOADS:
        if w["name"] == name:
            return dict(w)
    raise KeyError(name)


def make_seqlens(B, Nk, seed):
    """Per-batch key counts, uniform integers in [max(1, Nk // 8), Nk], from
    their own generator (seeded 700000 + seed)."""
    g = torch.Generator("cpu").manual_seed(700000 + int(seed))
    lo = max(1, Nk // 8)
    return torch.randint(lo, Nk + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def decode_workload(name):
    """The decoding workload dict with this name."""
    for w in DECODE_WORKLOADS:
        if w["name"] == name:
            return dict(w)
    raise KeyError(name)


def workload(name):
    """The workload dict with this name (or index)."""
    if isinstance(name, int):
        return dict(WORKLOADS[name])
    for w in WORKLOADS:
        if w["name"] == name:
            return dict(w)
    raise KeyError(name)


def make_qkv(B, H, N, d, dtype="bf16", q_std=1.0, seed=0):
    """Q, K, V as CPU tensors [B, H, N, d] of the storage dtype.

    Draw order is Q, K, V from one generator, so a given seed always yields
    the same three tensors whatever is done with them afterwards.
    """
    g = torch.Generator("cpu").manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    if q_std != 1.0:
        q.mul_(q_std)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    t = DTYPES[dtype]
    return q.to(t), k.to(t), v.to(t)


def make_decode(B, H, Nq, Nk, d, dtype="bf16", seed=0, dv=None):
    """Decoding inputs: Q [B, H, Nq, d] and a cache K [B, H, Nk, d], V
    [B, H, Nk, dv] (dv defaults to d), drawn Q, K, V from one generator
    (seeded 900000 + seed), N(0,1), rounded."""
    g = torch.Generator("cpu").manual_seed(900000 + int(seed))
    t = DTYPES[dtype]
    q = torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, Nk, d if dv is None else dv), generator=g, dtype=torch.float32)
    return q.to(t), k.to(t), v.to(t)


def make_varlen(lens_q, lens_k, H, d, dtype="bf16", seed=0, dv=None):
    """Packed batch: Q [sum(lens_q), H, d], K [sum(lens_k), H, d], V
    [sum(lens_k), H, dv] token-major, N(0,1) from one generator (seeded
    800000 + seed), rounded; and the int32 offsets cu_q, cu_k [B + 1]."""
    g = torch.Generator("cpu").manual_seed(800000 + int(seed))
    t = DTYPES[dtype]
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    q = torch.randn((tq, H, d), generator=g, dtype=torch.float32)
    k = torch.randn((tk, H, d), generator=g, dtype=torch.float32)
    v = torch.randn((tk, H, d if dv is None else dv), generator=g, dtype=torch.float32)
    cu_q = torch.tensor([0] + list(itertools.accumulate(int(x) for x in lens_q)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(itertools.accumulate(int(x) for x in lens_k)), dtype=torch.int32)
    return q.to(t), k.to(t), v.to(t), cu_q, cu_k


def make_dout(B, H, N, d, dtype="bf16", seed=0):
    """An upstream gradient dO [B, H, N, d] (N(0,1), rounded to the storage
    dtype) from its own generator, seeded 500000 + seed so it never repeats
    the Q, K, V draws of the same seed."""
    g = torch.Generator("cpu").manual_seed(500000 + int(seed))
    return torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(DTYPES[dtype])


def make_workload_qkv(w):
    """Q, K, V for a workload dict from ``WORKLOADS``."""
    return make_qkv(w["B"], w["H"], w["N"], w["d"], w["dtype"], w["q_std"],
                    w["seed"])


def sample_rows(N, count, seed, include=()):
    """Sorted distinct row indices in [0, N): ``include`` plus ``count`` drawn."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    extra = torch.randint(0, max(N, 1), (count,), generator=g).tolist() if N else []
    rows = sorted({int(r) for r in list(include) + extra if 0 <= int(r) < N})
    return rows
