"""The widened entry points at their full benchmarked sizes, against the
float64 oracle, through the C ABI.

The ragged small shapes in the other test files meet every code path, but
in fewer units than one persistent round of the forward kernels (one CTA
per SM walking several units).  These tests run the launches the bench
times — many rounds, with ring and barrier phases carried from unit to
unit and units that see no key between full ones — and compare whole heads
plus seeded sampled rows (and sampled keys for dK and dV) with the oracle
("FlashAttention: The Matrix You Never Have to Write Down", section "Check
it": the exact float64 reference, at sizes where the result matters).

* dropout: fa_fwd_dropout / fa_bwd_dropout on B1 H16 N4096 d128 bf16 at
  p = 0.1 (two whole heads), and the forward on a causal d = 64 shape of
  512 units;
* queries against a longer key set: fa_fwd_kv / fa_bwd_kv on the benched
  prefill chunk (B4 H32, 2048 queries after 14336 cached keys, d128 bf16,
  bottom-right), also with dropout (fa_fwd_kv_dropout / fa_bwd_kv_dropout,
  p = 0.1), and the forward on the padded batch (B16 H16, 1024 queries, up
  to 2048 keys with seeded counts, d64 bf16);
* packed batches: fa_fwd_varlen / fa_bwd_varlen on the benched batch of 16
  sequences of 256 .. 4096 tokens (H16 d128 bf16, causal).

Tolerances are those of the other GPU tests: the forward bounds (times
256/t for O with dropout), LSE within 1e-3, and the gradient bounds
relative to the largest reference magnitude.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import exact_tiled_attention_14_gb300 as fa
import oracle
import seeded_inputs
from gpu_common import LSE_TOL, TOL, require_gpu
from test_gpu_backward import check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def status_ok():
    torch.cuda.synchronize()
    code, word = fa.fa_status()
    assert code == fa.FA_OK, f"device status {word:#x}"


def pmap(fn, items):
    """fn over items on host threads (the oracle's C calls release the GIL)."""
    with ThreadPoolExecutor(max_workers=min(8, max(1, len(items)))) as ex:
        return list(ex.map(fn, items))


def check_rows(o, lse, o_ref, lse_ref, dtype, what, o_scale=1.0):
    """O and LSE rows of the CUDA path against the oracle's; rows the oracle
    leaves with no visible key must be exactly O = 0, LSE = -inf."""
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    empty = np.isneginf(lse_ref)
    assert np.all(np.isneginf(lse[empty])) and np.all(o[empty] == 0.0), f"{what}: empty rows"
    full = ~empty
    assert np.all(np.isfinite(o[full])) and np.all(np.isfinite(lse[full])), f"{what}: non-finite"
    err = np.abs(o[full] - o_ref[full])
    tmax, tmean = TOL[dtype]
    assert err.max() <= tmax * o_scale, f"{what}: max|dO| {err.max():.3e}"
    assert err.mean() <= tmean * o_scale, f"{what}: mean|dO| {err.mean():.3e}"
    lerr = np.abs(lse[full] - lse_ref[full]).max()
    assert lerr <= LSE_TOL, f"{what}: max|dLSE| {lerr:.3e}"
    print(f"{what}: max {err.max():.2e} mean {err.mean():.2e} lse {lerr:.2e}")


# ---------------------------------------------------------------- dropout

DROPOUT_CASES = [
    # name, B, H, N, d, dtype, causal, p, offset, heads compared whole
    ("b1_h16_n4096_d128_bf16_p0.1", 1, 16, 4096, 128, "bf16", False, 0.1, 3, [0, 15]),
    ("b1_h32_n4096_d64_fp16_causal_p0.1", 1, 32, 4096, 64, "fp16", True, 0.1, 9, [0, 31]),
]


@pytest.mark.parametrize("case", DROPOUT_CASES, ids=[c[0] for c in DROPOUT_CASES])
def test_dropout_forward_full_size(case):
    name, B, H, N, d, dtype, causal, p, off, heads = case
    seed = 1001
    q, k, v = seeded_inputs.make_qkv(B, H, N, d, dtype, 1.0, seed=seed)
    scale = d ** -0.5
    o, lse = fa.attention_forward_dropout(q.cuda(), k.cuda(), v.cuda(), p, seed, off,
                                          causal=causal, scale=scale)
    status_ok()
    o, lse = o.cpu().double().numpy(), lse.cpu().double().numpy()

    def ref(h):
        return oracle.attention_dropout(q[0, h].double().numpy(), k[0, h].double().numpy(),
                                        v[0, h].double().numpy(), h, seed, off, p,
                                        causal=causal, scale=scale)
    s = 256.0 / oracle.dropout_threshold(p)
    for h, (o_ref, l_ref) in zip(heads, pmap(ref, heads)):
        check_rows(o[0, h], lse[0, h], o_ref, l_ref, dtype, f"{name} head {h}", o_scale=s)


def test_dropout_backward_full_size():
    name, B, H, N, d, dtype, causal, p, off, heads = DROPOUT_CASES[0]
    seed = 1001
    q, k, v = seeded_inputs.make_qkv(B, H, N, d, dtype, 1.0, seed=seed)
    dout = seeded_inputs.make_dout(B, H, N, d, dtype, seed=seed)
    scale = d ** -0.5
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    o, lse = fa.attention_forward_dropout(dq_, dk_, dv_, p, seed, off, causal=causal, scale=scale)
    gq, gk, gv = fa.attention_backward_dropout(dq_, dk_, dv_, o, lse, do_, p, seed, off,
                                               causal=causal, scale=scale)
    status_ok()
    gq, gk, gv = gq.cpu(), gk.cpu(), gv.cpu()

    def ref(h):
        return oracle.attention_dropout_grad(q[0, h].double().numpy(), k[0, h].double().numpy(),
                                             v[0, h].double().numpy(), dout[0, h].double().numpy(),
                                             h, seed, off, p, causal=causal, scale=scale)
    for h, (rq, rk, rv) in zip(heads, pmap(ref, heads)):
        check_grad(f"{name} dQ head {h}", gq[0, h], rq, dtype)
        check_grad(f"{name} dK head {h}", gk[0, h], rk, dtype)
        check_grad(f"{name} dV head {h}", gv[0, h], rv, dtype)


# ---------------------------------------------------------------- kv

def kv_inputs(w):
    q, k, v = seeded_inputs.make_decode(w["B"], w["H"], w["Nq"], w["Nk"], w["d"], w["dtype"],
                                        seed=w["seed"])
    seqlens = seeded_inputs.make_seqlens(w["B"], w["Nk"], w["seed"]) if w["padded"] else None
    return q, k, v, seqlens


def kv_offset(w, n):
    return n - w["Nq"] if w["causal"] == "bottom_right" else 0


def kv_len(w, seqlens, b):
    return w["Nk"] if seqlens is None else max(0, min(int(seqlens[b]), w["Nk"]))


@pytest.mark.parametrize("name", [w["name"] for w in seeded_inputs.KV_WORKLOADS])
def test_kv_forward_full_size(name):
    w = seeded_inputs.kv_workload(name)
    B, H, Nq = w["B"], w["H"], w["Nq"]
    q, k, v, seqlens = kv_inputs(w)
    sl = None if seqlens is None else seqlens.cuda()
    o, lse = fa.attention_forward_kv(q.cuda(), k.cuda(), v.cuda(), causal=w["causal"],
                                     seqlens_k=sl, scale=w["scale"])
    status_ok()
    o, lse = o.cpu().double().numpy(), lse.cpu().double().numpy()
    # whole heads: the first and the last (batch, head), and for a padded
    # batch one head of every batch; seeded rows of twelve more heads
    whole = {(0, 0), (B - 1, H - 1)}
    if w["padded"]:
        whole |= {(b, (3 * b) % H) for b in range(B)}
    g = torch.Generator("cpu").manual_seed(w["seed"])
    sampled = {(int(torch.randint(0, B, (1,), generator=g)), int(torch.randint(0, H, (1,), generator=g)))
               for _ in range(12)} - whole
    edges = (0, 1, 127, 128, 255, 256, Nq // 2, Nq - 129, Nq - 128, Nq - 1)
    jobs = [(b, h, np.arange(Nq)) for b, h in sorted(whole)]
    jobs += [(b, h, np.asarray(seeded_inputs.sample_rows(Nq, 24, seed=b * H + h, include=edges)))
             for b, h in sorted(sampled)]

    def ref(job):
        b, h, rows = job
        n = kv_len(w, seqlens, b)
        pos = rows.astype(np.int64) + kv_offset(w, n)
        return oracle.attention_rows(q[b, h, rows].double().numpy(), pos,
                                     k[b, h, :n].double().numpy(), v[b, h, :n].double().numpy(),
                                     causal=w["causal"] is not None, scale=w["scale"])
    for (b, h, rows), (o_ref, l_ref) in zip(jobs, pmap(ref, jobs)):
        check_rows(o[b, h, rows], lse[b, h, rows], o_ref, l_ref, w["dtype"],
                   f"{name} ({b},{h}) {len(rows)} rows")


def test_kv_backward_full_size():
    w = seeded_inputs.kv_workload(seeded_inputs.KV_WORKLOADS[0]["name"])
    B, H, Nq, Nk = w["B"], w["H"], w["Nq"], w["Nk"]
    q, k, v, seqlens = kv_inputs(w)
    assert seqlens is None
    dout = seeded_inputs.make_dout(B, H, Nq, w["d"], w["dtype"], seed=w["seed"])
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    o, lse = fa.attention_forward_kv(dq_, dk_, dv_, causal=w["causal"], scale=w["scale"])
    gq, gk, gv = fa.attention_backward_kv(dq_, dk_, dv_, o, lse, do_, causal=w["causal"],
                                          scale=w["scale"])
    status_ok()
    gq, gk, gv = gq.cpu(), gk.cpu(), gv.cpu()
    off = kv_offset(w, Nk)
    keys = np.asarray(seeded_inputs.sample_rows(
        Nk, 192, seed=w["seed"],
        include=(0, 1, 127, 128, off - 1, off, off + 1, off + 127, off + 128, Nk - 129, Nk - 128,
                 Nk - 1)), dtype=np.int64)
    heads = [(0, 0), (B - 1, H - 1)]

    def ref(bh):
        b, h = bh
        qh, gh = q[b, h].double().numpy(), dout[b, h].double().numpy()
        kh, vh = k[b, h].double().numpy(), v[b, h].double().numpy()
        pos = np.arange(Nq, dtype=np.int64) + off
        rq, l_ref, delta = oracle.grad_query_rows(qh, gh, pos, kh, vh, causal=True,
                                                  scale=w["scale"])
        rk, rv = oracle.grad_key_rows(kh[keys], vh[keys], keys - off, qh, gh, l_ref, delta,
                                      causal=True, scale=w["scale"])
        return rq, rk, rv
    for (b, h), (rq, rk, rv) in zip(heads, pmap(ref, heads)):
        what = f"{w['name']} ({b},{h})"
        check_grad(what + " dQ", gq[b, h], rq, w["dtype"])
        check_grad(what + " dK", gk[b, h][keys], rk, w["dtype"])
        check_grad(what + " dV", gv[b, h][keys], rv, w["dtype"])


def test_kv_dropout_full_size():
    """fa_fwd_kv_dropout / fa_bwd_kv_dropout on the benched prefill chunk at
    p = 0.1 (the d = 128 mask generator warpgroup over 1024 units): O, LSE,
    dQ, dK and dV of the first and last (batch, head), each query at its
    position after the cache, the mask drawn by (batch * head, row, key)."""
    w = seeded_inputs.kv_workload(seeded_inputs.KV_WORKLOADS[0]["name"])
    B, H, Nq, Nk = w["B"], w["H"], w["Nq"], w["Nk"]
    q, k, v, seqlens = kv_inputs(w)
    assert seqlens is None
    p, seed, off = 0.1, 2024, 7
    dout = seeded_inputs.make_dout(B, H, Nq, w["d"], w["dtype"], seed=w["seed"] + 1)
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    o, lse = fa.attention_forward_kv(dq_, dk_, dv_, causal=w["causal"], scale=w["scale"],
                                     dropout_p=p, seed=seed, offset=off)
    gq, gk, gv = fa.attention_backward_kv(dq_, dk_, dv_, o, lse, do_, causal=w["causal"],
                                          scale=w["scale"], dropout_p=p, seed=seed, offset=off)
    status_ok()
    o, lse = o.cpu().double().numpy(), lse.cpu().double().numpy()
    gq, gk, gv = gq.cpu(), gk.cpu(), gv.cpu()
    shift = kv_offset(w, Nk)
    heads = [(0, 0), (B - 1, H - 1)]

    def ref(bh):
        b, h = bh
        args = (q[b, h].double().numpy(), k[b, h].double().numpy(), v[b, h].double().numpy())
        fwd = oracle.attention_dropout(*args, b * H + h, seed, off, p, causal=True,
                                       scale=w["scale"], q_offset=shift)
        grad = oracle.attention_dropout_grad(*args, dout[b, h].double().numpy(), b * H + h, seed,
                                             off, p, causal=True, scale=w["scale"], q_offset=shift)
        return fwd, grad
    s = 256.0 / oracle.dropout_threshold(p)
    for (b, h), ((o_ref, l_ref), (rq, rk, rv)) in zip(heads, pmap(ref, heads)):
        what = f"{w['name']} p={p} ({b},{h})"
        check_rows(o[b, h], lse[b, h], o_ref, l_ref, w["dtype"], what, o_scale=s)
        check_grad(what + " dQ", gq[b, h], rq, w["dtype"])
        check_grad(what + " dK", gk[b, h], rk, w["dtype"])
        check_grad(what + " dV", gv[b, h], rv, w["dtype"])


# ---------------------------------------------------------------- packed batches

def varlen_inputs(w):
    lens = seeded_inputs.varlen_lengths(w["B"], w["lo"], w["hi"], w["seed"])
    q, k, v, cu_q, cu_k = seeded_inputs.make_varlen(lens, lens, w["H"], w["d"], w["dtype"],
                                                    seed=w["seed"])
    return lens, q, k, v, cu_q, cu_k


def test_varlen_forward_full_size():
    w = seeded_inputs.varlen_workload(seeded_inputs.VARLEN_WORKLOADS[0]["name"])
    H = w["H"]
    lens, q, k, v, cu_q, cu_k = varlen_inputs(w)
    o, lse = fa.attention_forward_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(),
                                         max(lens), causal=w["causal"], scale=w["scale"])
    status_ok()
    o, lse = o.cpu().double().numpy(), lse.cpu().double().numpy()
    cu = cu_q.tolist()
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    # every head of the longest and the shortest sequence whole; two heads of
    # every other sequence on seeded rows and the tile edges
    jobs = [(b, h, np.arange(lens[b])) for b in (longest, shortest) for h in range(H)]
    for b in range(len(lens)):
        if b in (longest, shortest):
            continue
        n = lens[b]
        rows = np.asarray(seeded_inputs.sample_rows(
            n, 32, seed=b, include=(0, 127, 128, 255, 256, n - 129, n - 128, n - 1)))
        jobs += [(b, b % H, rows), (b, (b + 7) % H, rows)]

    def ref(job):
        b, h, rows = job
        s0, s1 = cu[b], cu[b + 1]
        return oracle.attention_rows(q[s0 + rows, h].double().numpy(), rows.astype(np.int64),
                                     k[s0:s1, h].double().numpy(), v[s0:s1, h].double().numpy(),
                                     causal=True, scale=w["scale"])
    for (b, h, rows), (o_ref, l_ref) in zip(jobs, pmap(ref, jobs)):
        s0 = cu[b]
        check_rows(o[s0 + rows, h], lse[h, s0 + rows], o_ref, l_ref, w["dtype"],
                   f"sequence {b} (len {lens[b]}) head {h}: {len(rows)} rows")


def test_varlen_backward_full_size():
    w = seeded_inputs.varlen_workload(seeded_inputs.VARLEN_WORKLOADS[0]["name"])
    H = w["H"]
    lens, q, k, v, cu_q, cu_k = varlen_inputs(w)
    total = sum(lens)
    g = torch.Generator("cpu").manual_seed(500000 + w["seed"])
    dout = torch.randn((total, H, w["d"]), generator=g).to(q.dtype)
    dq_, dk_, dv_, do_ = (t.cuda() for t in (q, k, v, dout))
    dcq, dck = cu_q.cuda(), cu_k.cuda()
    o, lse = fa.attention_forward_varlen(dq_, dk_, dv_, dcq, dck, max(lens), causal=w["causal"],
                                         scale=w["scale"])
    gq, gk, gv = fa.attention_backward_varlen(dq_, dk_, dv_, o, lse, do_, dcq, dck, max(lens),
                                              max(lens), causal=w["causal"], scale=w["scale"])
    status_ok()
    gq, gk, gv = gq.cpu(), gk.cpu(), gv.cpu()
    cu = cu_q.tolist()
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    jobs = [(longest, 0), (longest, H - 1), (shortest, 3), ((longest + 1) % len(lens), 5)]

    def ref(job):
        b, h = job
        s0, s1 = cu[b], cu[b + 1]
        n = s1 - s0
        qh, gh = q[s0:s1, h].double().numpy(), dout[s0:s1, h].double().numpy()
        kh, vh = k[s0:s1, h].double().numpy(), v[s0:s1, h].double().numpy()
        rq, l_ref, delta = oracle.grad_query_rows(qh, gh, np.arange(n, dtype=np.int64), kh, vh,
                                                  causal=True, scale=w["scale"])
        keys = np.asarray(seeded_inputs.sample_rows(
            n, 128, seed=b * H + h, include=(0, 1, 127, 128, n - 129, n - 128, n - 1)),
            dtype=np.int64)
        rk, rv = oracle.grad_key_rows(kh[keys], vh[keys], keys, qh, gh, l_ref, delta,
                                      causal=True, scale=w["scale"])
        return keys, rq, rk, rv
    for (b, h), (keys, rq, rk, rv) in zip(jobs, pmap(ref, jobs)):
        s0, s1 = cu[b], cu[b + 1]
        what = f"sequence {b} (len {lens[b]}) head {h}"
        check_grad(what + " dQ", gq[s0:s1, h], rq, w["dtype"])
        check_grad(what + " dK", gk[s0 + keys, h], rk, w["dtype"])
        check_grad(what + " dV", gv[s0 + keys, h], rv, w["dtype"])
