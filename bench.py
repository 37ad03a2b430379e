#!/usr/bin/env python3
"""Forward-attention benchmark on GB300: TFLOP/s and the fraction of the
dense BF16 tensor-core peak.

One step = one exact-attention forward pass (one ``fa_fwd`` launch) over one
synthetic workload already resident in device memory.  FLOPs per step follow
the usual convention 4*B*H*N^2*d (two matmuls of 2*N^2*d each), halved for
causal masking.

Default workload: the largest of the five synthetic workloads, B=4, H=32,
N=8192, d=128, bf16, causal, seeded inputs.  ``--workload`` selects another.

Timing: one pass times exactly ``--steps`` steps (CUDA events around each
launch on the launching stream, a barrier and a device synchronise on both
sides); passes repeat back to back until ``--min-timed-ms`` (default 1000)
of device time is covered, so the clock sampler sees the GPU under load for
at least that long.  The line reports ``timed_passes``; value and
ms_per_step cover all passes.

Printed (rank 0, one JSON line): value (whole job TFLOP/s), ms_per_step,
``roofline`` (achieved vs the measured bf16 peak; DRAM traffic from the last
ncu capture when the kernel sources still match it), ``cpu_baseline`` (the
float64 oracle timed on the host cores on a bounded sample of rows), ``e2e``
(same metric through the public call with pinned host buffers, copies in the
timed region), ``clocks`` (nvidia-smi samples during the timed region) and
``gpu_launches``.

``--impl reference`` times the float64 oracle on the host cores instead
(rank 0 only), on bounded samples of the same workload.

``--pass decode`` times split-KV decoding (``fa_decode``) on a decoding
workload (GB/s of K/V read against the measured HBM copy bandwidth).

``--pass kv`` times ``fa_fwd_kv`` (queries against a key set of another
length, with padding and causal alignment) on a kv workload; FLOPs are 4 d
per visible (query, key) pair.

``--pass varlen`` times ``fa_fwd_varlen`` on a packed batch of sequences of
mixed lengths (and, for context, the same batch padded through
``fa_fwd_kv``).

``--dropout P`` times ``fa_fwd_dropout`` (or ``fa_bwd_dropout`` with
``--pass bwd``): the mask drawn on the device from (seed, offset), a new
offset per forward step.

``--pass bwd`` times the backward pass instead: one step = one ``fa_bwd``
call (two kernels: the D pass and the dK/dV + dQ grid) with the forward's O
and LSE and a seeded dO resident on the device; FLOPs are 2.5x the
forward's (five matmuls against two).  ``--onepass`` times
``fa_bwd_onepass`` instead (the D pass, one grid that also sums dQ through
an fp32 workspace, and the dQ conversion).

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
forward pass has no exchange step); value = all ranks' FLOPs / the slowest
rank's time.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
DEFAULT_WORKLOAD = "b4_h32_n8192_d128_bf16_causal"
METRIC = "attention fwd TFLOP/s (causal halved) and % of GB300 dense BF16 tensor peak"
METRIC_DEC = "attention decode (split-KV) K/V read GB/s and % of GB300 HBM copy bandwidth"
METRIC_BWD = ("attention bwd TFLOP/s (2.5x the forward's FLOPs, causal halved) and % of GB300 "
              "dense BF16 tensor peak")
METRIC_KV = ("attention fwd, queries against a key set of another length: TFLOP/s (4 d per "
             "visible query-key pair) and % of GB300 dense BF16 tensor peak")
METRIC_VARLEN = ("attention fwd over a packed variable-length batch: TFLOP/s (4 d per visible "
                 "query-key pair) and % of GB300 dense BF16 tensor peak")
FALLBACK_PEAK_TFLOPS = 1900.0


# ---------------------------------------------------------------- accounting

def step_flops(w):
    f = 4.0 * w["B"] * w["H"] * w["N"] * w["N"] * w["d"]
    return f / 2 if w["causal"] else f


def step_flops_bwd(w):
    """Backward FLOPs by the usual convention: five N^2 d matmuls (dV, dP, dQ, dK
    and the recomputed S) against the forward's two, i.e. 2.5x the forward."""
    return 2.5 * step_flops(w)


def io_bytes_bwd(w):
    elems = w["B"] * w["H"] * w["N"] * w["d"]
    rows = w["B"] * w["H"] * w["N"]
    return dict(h2d=5 * elems * 2 + rows * 4, d2h=3 * elems * 2)


def io_bytes(w):
    elems = w["B"] * w["H"] * w["N"] * w["d"]
    return dict(h2d=3 * elems * 2, d2h=elems * 2 + w["B"] * w["H"] * w["N"] * 4)


def kv_positions(w, seqlens):
    """Per batch: (key count, position of query row 0) of an fa_fwd_kv workload."""
    out = []
    for b in range(w["B"]):
        n = w["Nk"] if seqlens is None else max(0, min(int(seqlens[b]), w["Nk"]))
        out.append((n, n - w["Nq"] if w["causal"] == "bottom_right" else 0))
    return out


def kv_visible_pairs(w, n, off):
    """(query, key) pairs of one head that the mask leaves visible: the
    forward's FLOP count is 4 d per visible pair (the square causal
    convention N^2/2 is this count up to the N/2 diagonal term)."""
    Nq = w["Nq"]
    if not w["causal"]:
        return Nq * n
    # row i sees min(n, max(0, i + off + 1)) keys: rows [lo, hi) see a partial
    # prefix, rows from `full` on see all n keys
    lo = max(0, -off)
    hi = min(Nq, n - off - 1)
    total = 0
    if hi > lo:
        total += (hi - lo) * (off + 1) + (hi * (hi - 1) - lo * (lo - 1)) // 2
    full = max(lo, n - off - 1)
    if Nq > full:
        total += (Nq - full) * n
    return total


def step_flops_kv(w, seqlens):
    return sum(4.0 * w["d"] * w["H"] * kv_visible_pairs(w, n, off)
               for n, off in kv_positions(w, seqlens))


def kernel_source_hash():
    """Hash of the sources the forward kernel and its launch are built from; a
    stored ncu traffic figure is only valid for it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_14_gb300", "csrc")
    for name in FORWARD_SOURCES:
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


# The forward kernel, its launch and the host code that shapes it (checks,
# descriptors, unit order); the backward and decoding entry points live in
# other files and do not move the forward's DRAM traffic.
FORWARD_SOURCES = ("fa_common.cu", "fa_fwd_api.cu", "fa_host.cuh", "fa_fwd_d128.cu",
                   "fa_fwd_d64.cu", "fa_fwd_kernel.cuh", "fa_launch.cuh", "ptx_sm103.cuh")


def stored_traffic(workload):
    """DRAM bytes per launch from profiles/traffic.json, if taken on these sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        data = json.load(open(path))
    except (OSError, ValueError):
        return None, "no profiles/traffic.json"
    entry = data.get("workloads", {}).get(workload)
    if not entry:
        return None, "no ncu capture for this workload"
    if entry.get("kernel_hash") != kernel_source_hash():
        return None, "kernel changed since the ncu capture"
    return entry.get("dram_bytes_per_launch"), entry.get("note")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        data = json.load(open(path))
        return float(data["bf16_tflops"]), float(data.get("bf16_tflops_sustained") or 0), "measured"
    except (OSError, ValueError, KeyError, TypeError):
        return FALLBACK_PEAK_TFLOPS, 1700.0, "fallback"


def dtype_peak_check(device):
    """cuBLAS dense-GEMM rates of fp16 and bf16 at 8192^3 on this GPU (a few
    timed products each, after a warm-up): fp16 workloads take the measured
    bf16 peak times the nominal fp16/bf16 ratio of 1, and this probe, run
    after the timed region, shows that ratio on the box."""
    import torch
    out = {}
    n = 8192
    for name, dt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
        g = torch.Generator(device=device).manual_seed(7)
        a = torch.randn(n, n, device=device, dtype=dt, generator=g)
        b = torch.randn(n, n, device=device, dtype=dt, generator=g)
        for _ in range(3):
            torch.matmul(a, b)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        s.record()
        for _ in range(10):
            torch.matmul(a, b)
        e.record()
        torch.cuda.synchronize(device)
        out[name + "_tflops"] = 10 * 2.0 * n ** 3 / (s.elapsed_time(e) * 1e-3) / 1e12
        del a, b
    out["fp16_over_bf16"] = out["fp16_tflops"] / out["bf16_tflops"]
    out["probe"] = "torch.matmul 8192^3, 10 products after 3 warm-up, cuBLAS, outside the timed region"
    return out


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock, power and clock-event reasons sampled while the benchmark runs.

    Polls NVML (read-only queries through ctypes) every ~2 ms in a thread;
    falls back to ``nvidia-smi -lms 20`` when NVML cannot be opened.
    """

    # NVML clock-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.sw_power_cap",
                  "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown"]

    def __init__(self, device_index):
        self.samples = []        # (host time, sm_mhz, max_mhz, power_w, reason names)
        self.error = None
        self.source = None
        self.device_index = device_index
        self._stop = threading.Event()
        self.thread = None
        self.proc = None

    # -- NVML
    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        ok = False
        try:
            props = torch.cuda.get_device_properties(self.device_index)
            bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(handle)) == 0
        except Exception:
            ok = False
        if not ok:
            count = ctypes.c_uint(0)
            lib.nvmlDeviceGetCount_v2(ctypes.byref(count))
            if count.value != 1:
                raise OSError("cannot identify the GPU in NVML")
            if lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(handle)) != 0:
                raise OSError("nvmlDeviceGetHandleByIndex failed")
        return lib, handle

    def _nvml_loop(self, lib, handle):
        import ctypes
        clk, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            t = time.time()
            if lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0:
                lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))
                p = lib.nvmlDeviceGetPowerUsage(handle, ctypes.byref(pw))
                get_reasons(handle, ctypes.byref(rs))
                names = [n for bit, n in self.REASONS.items() if rs.value & bit]
                self.samples.append((t, float(clk.value), float(mx.value),
                                     pw.value / 1000.0 if p == 0 else None, names))
            time.sleep(0.002)

    # -- nvidia-smi fallback
    def _smi_loop(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.SMI_FIELDS):
                continue
            try:
                names = [n for n, v in zip(["sw_power_cap", "hw_slowdown", "sw_thermal_slowdown",
                                            "hw_thermal_slowdown"], parts[3:])
                         if v.lower() == "active"]
                pw = float(parts[2]) if parts[2] not in ("[N/A]", "") else None
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), pw, names))
            except ValueError:
                pass

    def start(self):
        try:
            lib, handle = self._nvml_open()
            self.source = "nvml"
            self.thread = threading.Thread(target=self._nvml_loop, args=(lib, handle), daemon=True)
        except OSError as e:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=" + ",".join(self.SMI_FIELDS),
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = f"nvidia-smi ({e})"
                self.thread = threading.Thread(target=self._smi_loop, daemon=True)
            except OSError as e2:
                self.error = f"no clock source: {e}; {e2}"
                return self
        self.thread.start()
        return self

    def stop(self):
        self._stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1, fallback_window=None):
        def pick(a, b):
            return [x for x in self.samples if a <= x[0] <= b]
        window = "timed"
        rows = pick(t0, t1)
        if len(rows) < 3 and fallback_window:
            rows, window = pick(*fallback_window), "warmup+timed"
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": len(rows),
               "window": window, "source": self.source}
        if self.error:
            out["error"] = self.error
        if not rows:
            return out
        out["sm_mhz"] = statistics.median(r[1] for r in rows)
        out["sm_min_mhz"] = min(r[1] for r in rows)
        out["sm_max_mhz"] = max(r[2] for r in rows)
        pws = [r[3] for r in rows if r[3] is not None]
        if pws:
            out["power_w_max"] = max(pws)
        out["reasons"] = sorted({n for r in rows for n in r[4]})
        return out


# ---------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(x, world, device=None):
    """Largest value of x over all ranks (x itself when running alone)."""
    if world == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world, device=None):
    if world > 1:
        if device is not None and device.type == "cuda":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample(w, q, k, v, budget_s, start_head=0):
    """Time the float64 oracle on whole heads of the workload for about budget_s.

    Heads are taken in order from ``start_head`` (wrapping) until the budget
    is spent or every head is done.  Every head does the same work, so the
    throughput of whole heads is the throughput of the workload.  Returns
    (TFLOP/s, seconds, heads, cores, description).
    """
    import oracle
    lib = oracle.load()
    B, H = w["B"], w["H"]
    nheads = B * H
    cores = oracle.num_threads(lib)
    done, spent = 0, 0.0
    while done < nheads and (done == 0 or spent < budget_s):
        hb = (start_head + done) % nheads
        b, h = divmod(hb, H)
        qh, kh, vh = (t[b, h].double().numpy() for t in (q, k, v))
        t0 = time.perf_counter()
        oracle.attention(qh, kh, vh, causal=w["causal"], scale=w["scale"], lib=lib)
        spent += time.perf_counter() - t0
        done += 1
    flops = step_flops(w) * done / nheads
    desc = (f"{done} of {nheads} whole heads of {w['name']} (float64, {cores} threads); "
            "every head does the same work")
    return flops / spent / 1e12, spent, done, cores, desc


def oracle_grad_sample(w, q, k, v, dout, budget_s, start_head=0):
    """Time the float64 gradient oracle on whole heads for about budget_s
    (the backward counterpart of ``oracle_sample``)."""
    import oracle
    lib = oracle.load()
    B, H = w["B"], w["H"]
    nheads = B * H
    cores = oracle.num_threads(lib)
    done, spent = 0, 0.0
    while done < nheads and (done == 0 or spent < budget_s):
        hb = (start_head + done) % nheads
        b, h = divmod(hb, H)
        qh, kh, vh, gh = (t[b, h].double().numpy() for t in (q, k, v, dout))
        t0 = time.perf_counter()
        oracle.attention_grad(qh, kh, vh, gh, causal=w["causal"], scale=w["scale"], lib=lib)
        spent += time.perf_counter() - t0
        done += 1
    flops = step_flops_bwd(w) * done / nheads
    desc = (f"gradients of {done} of {nheads} whole heads of {w['name']} (float64, {cores} "
            "threads); every head does the same work")
    return flops / spent / 1e12, spent, done, cores, desc


def dropout_oracle_sample(w, q, k, v, dout, p, budget_s):
    """Time the float64 dropout oracle (forward, or gradients when ``dout``
    is given) on whole heads for about budget_s; one thread per head."""
    import oracle
    lib = oracle.load()
    B, H = w["B"], w["H"]
    done, spent = 0, 0.0
    while done < B * H and (done == 0 or spent < budget_s):
        b, h = divmod(done, H)
        qh, kh, vh = (t[b, h].double().numpy() for t in (q, k, v))
        t0 = time.perf_counter()
        if dout is None:
            oracle.attention_dropout(qh, kh, vh, done, w["seed"], 0, p, causal=w["causal"],
                                     scale=w["scale"], lib=lib)
        else:
            oracle.attention_dropout_grad(qh, kh, vh, dout[b, h].double().numpy(), done,
                                          w["seed"], 0, p, causal=w["causal"], scale=w["scale"],
                                          lib=lib)
        spent += time.perf_counter() - t0
        done += 1
    per_head = (step_flops(w) if dout is None else step_flops_bwd(w)) / (B * H)
    desc = (f"{done} of {B * H} whole heads of {w['name']} with dropout {p} (float64, one "
            "thread); every head does the same work")
    return per_head * done / spent / 1e12, spent, done, 1, desc


def timed_region(step, steps, min_ms, stream, world, device, max_passes=1000):
    """The timed region of a bench arm.

    One pass times exactly ``steps`` calls of ``step(i)`` with a CUDA event
    pair around each call on ``stream``, bracketed by a barrier and a device
    synchronise on both sides.  Passes follow each other until the device
    time of all passes (the slowest rank's, so every rank stops after the
    same pass) reaches ``min_ms``: with a short step the GPU then runs under
    load long enough for the clock sampler to see it.  Step indices keep
    counting across passes (input replicas and dropout offsets rotate on).

    Returns (total device ms over all passes, list of per-step ms, passes,
    host time at the start, host time at the end).
    """
    total_ms, per_step, passes = 0.0, [], 0
    t0 = None
    while True:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier(world, device)
        torch.cuda.synchronize()
        if t0 is None:
            t0 = time.time()
        for i in range(steps):
            starts[i].record(stream)
            step(passes * steps + i)
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier(world, device)
        total_ms += max_over_ranks(starts[0].elapsed_time(ends[-1]), world, device)
        per_step += [a.elapsed_time(b) for a, b in zip(starts, ends)]
        passes += 1
        if total_ms >= min_ms or passes >= max_passes:
            break
    return total_ms, per_step, passes, t0, time.time()


def time_launches(fn, reps, warmup=3):
    """Mean milliseconds of fn() over reps launches (CUDA events on the
    current stream, after warmup calls)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def backward_line(ms, flops, entry, peak):
    """The "backward" object of a kv or varlen bench line: one call of the
    backward entry point on the same workload, 2.5x the forward's FLOPs."""
    return {"entry": entry, "ms": ms, "tflops": 2.5 * flops / (ms * 1e-3) / 1e12,
            "frac": 2.5 * flops / (ms * 1e-3) / 1e12 / peak,
            "flops_per_launch": 2.5 * flops, "scope": "D pass and the dK/dV + dQ grid"}


def graph_replay(launch, n_launch, reps):
    """Milliseconds per launch when ``launch(i, stream)`` is captured
    n_launch times into one CUDA graph and the graph is replayed ``reps``
    times (CUDA events around the replays)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(3):
            launch(i, side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for i in range(n_launch):
            launch(i, cs)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * n_launch)


# ---------------------------------------------------------------- arms

def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v = seeded_inputs.make_workload_qkv(w)
    total = args.steps + args.warmup
    per_step = max(0.2, min(10.0, args.reference_seconds / max(total, 1)))
    import oracle
    oracle.load()
    vals = []
    bwd = args.pass_ == "bwd"
    dout = seeded_inputs.make_dout(w["B"], w["H"], w["N"], w["d"], w["dtype"], seed=w["seed"]) \
        if bwd else None
    for i in range(total):
        if args.dropout > 0:
            tf, dt, heads, cores, desc = dropout_oracle_sample(w, q, k, v, dout, args.dropout,
                                                               per_step)
        elif bwd:
            tf, dt, heads, cores, desc = oracle_grad_sample(w, q, k, v, dout, per_step, start_head=i)
        else:
            tf, dt, heads, cores, desc = oracle_sample(w, q, k, v, per_step, start_head=i)
        if i >= args.warmup:
            vals.append((tf, dt))
    value = statistics.median(tf for tf, _ in vals)
    ms = statistics.median(dt for _, dt in vals) * 1e3
    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": "TFLOP/s",
        "impl": "reference", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["name"], "B": w["B"], "H": w["H"], "N": w["N"], "d": w["d"],
                   "causal": w["causal"], "storage_dtype": w["dtype"], "seed": w["seed"],
                   "pass": "backward" if bwd else "forward", "dropout": args.dropout},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_kv(args, w):
    """Reference arm of ``--pass kv``: the float64 oracle on the host cores,
    bounded samples of whole (batch, head) pairs per step (rank 0 only)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v = seeded_inputs.make_decode(w["B"], w["H"], w["Nq"], w["Nk"], w["d"], w["dtype"],
                                        seed=w["seed"])
    seqlens = seeded_inputs.make_seqlens(w["B"], w["Nk"], w["seed"]) if w["padded"] else None
    total = args.steps + args.warmup
    per_step = max(0.2, min(10.0, args.reference_seconds / max(total, 1)))
    vals = []
    for i in range(total):
        tf, dt, heads, cores, desc = kv_oracle_sample(w, q, k, v, seqlens, per_step, start_head=i)
        if i >= args.warmup:
            vals.append((tf, dt))
    value = statistics.median(tf for tf, _ in vals)
    line = {
        "metric": METRIC_KV, "value": value, "unit": "TFLOP/s", "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(dt for _, dt in vals) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["name"], "pass": "kv", "B": w["B"], "H": w["H"], "Nq": w["Nq"],
                   "Nk": w["Nk"], "d": w["d"], "causal": w["causal"], "storage_dtype": w["dtype"],
                   "seed": w["seed"]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def e2e_pipelined(fa, w, q, k, v, bufs, ws, drop, stream, device, steps, world):
    """Milliseconds per step of the forward pass end to end through the
    public call (``attention_forward``), from pinned host inputs to pinned
    host outputs, with consecutive steps overlapped over two device buffer
    sets (uploads of q, k, v each on a stream of its own, compute, downloads);
    every step copies its own inputs in and its outputs out."""
    B, H, N = w["B"], w["H"], w["N"]
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    sets = [bufs[0]]
    if len(bufs) > 1:
        sets.append(bufs[1])
    else:
        dq2, dk2, dv2 = (torch.empty_like(t) for t in bufs[0][:3])
        sets.append((dq2, dk2, dv2, torch.empty_like(bufs[0][3]), torch.empty_like(bufs[0][4])))
    hos = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(2)]
    hls = [torch.empty((B, H, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    s_ins = [torch.cuda.Stream(device) for _ in range(3)]   # one upload stream per input
    s_out = torch.cuda.Stream(device)
    ev_in = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(i):
        b = i & 1
        dq, dk, dv, o, lse = sets[b]
        for s_in, ev, dst, src in zip(s_ins, ev_in[b], (dq, dk, dv), (hq, hk, hv)):
            if used[b]:
                s_in.wait_event(ev_comp[b])    # the compute of step i-2 has read these inputs
            with torch.cuda.stream(s_in):
                dst.copy_(src, non_blocking=True)
            ev.record(s_in)
            stream.wait_event(ev)
        if used[b]:
            stream.wait_event(ev_out[b])       # step i-2's outputs have been read out
        if drop > 0:
            fa.attention_forward_dropout(dq, dk, dv, drop, w["seed"], 0, causal=w["causal"],
                                         scale=w["scale"], out=o, lse=lse, stream=stream)
        else:
            fa.attention_forward(dq, dk, dv, causal=w["causal"], scale=w["scale"], out=o,
                                 lse=lse, stream=stream, workspace=ws)
        ev_comp[b].record(stream)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            hos[b].copy_(o, non_blocking=True)
            hls[b].copy_(lse, non_blocking=True)
        ev_out[b].record(s_out)
        used[b] = True

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    barrier(world, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_in in s_ins:
        s_in.wait_stream(stream)
    for i in range(steps):
        step(i)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(e0.elapsed_time(e1) / steps, world, device)


def run_ours(args, w):
    import exact_tiled_attention_14_gb300 as fa

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    fa.load_library()

    sampler = ClockSampler(local).start()
    q, k, v = seeded_inputs.make_workload_qkv(w)
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    per_replica = io_bytes(w)["h2d"] + io_bytes(w)["d2h"]
    # Rotate through input replicas so a step never finds its inputs in L2
    # (capped for tiny workloads, which are launch-bound, not memory-bound).
    replicas = 1 if per_replica > 2 * L2_BYTES else int(math.ceil(2 * L2_BYTES / per_replica)) + 1
    replicas = min(replicas, 64)
    bufs = []
    for _ in range(replicas):
        dq, dk, dv = (t.to(device) for t in (q, k, v))
        o = torch.empty_like(dq)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
        bufs.append((dq, dk, dv, o, lse))
    stream = torch.cuda.current_stream(device)
    # Balancing workspace of fa_fwd_ws (allocated once, outside the timed
    # region); None when this shape leaves no partial last round.
    ws = fa.make_workspace(B, H, N, d, w["causal"], device=device) if args.split else None
    ws_bytes = 0 if ws is None else ws.numel()

    drop = args.dropout

    def launch(i, st):
        dq, dk, dv, o, lse = bufs[i % replicas]
        if drop > 0:
            rc = fa.fa_fwd_dropout(dq, dk, dv, o, lse, B, H, N, d, w["causal"], w["scale"], drop,
                                   w["seed"], i, fa.dtype_code(dq.dtype), st)
        elif ws is None:
            rc = fa.fa_fwd(dq, dk, dv, o, lse, B, H, N, d, w["causal"], w["scale"],
                           fa.dtype_code(dq.dtype), st)
        else:
            rc = fa.fa_fwd_ws(dq, dk, dv, o, lse, B, H, N, d, w["causal"], w["scale"],
                              fa.dtype_code(dq.dtype), ws, ws_bytes, st)
        if rc:
            raise fa.FaError(rc)

    def step(i):
        launch(i, stream)

    t_warm = time.time()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    code, word = fa.fa_status(stream)
    if code:
        raise fa.FaError(code, f"warmup status {word:#x}")

    total_ms, per_step, passes, t0, t1 = timed_region(step, args.steps, args.min_timed_ms, stream,
                                                      world, device)
    kern_ms = statistics.mean(per_step)
    code, word = fa.fa_status(stream)
    if code:
        raise fa.FaError(code, f"timed status {word:#x}")
    kern_ms_max = max_over_ranks(kern_ms, world, device)
    # launch-bound workloads: also the per-launch time of CUDA-graph replay
    # (100 launches captured once, the graph replayed 10 times)
    graph = graph_replay(launch, 100, 10) if kern_ms < 0.05 else None

    # ---- end to end: pinned host inputs -> device -> fa_fwd -> host outputs.
    # Consecutive steps are pipelined as a serving loop would run them: two
    # sets of device buffers, the host-to-device copies on one stream, the
    # attention call on another and the device-to-host copies on a third, so
    # step i+1's inputs upload and step i-1's outputs download while step i
    # computes.  Every step still copies all its inputs in and its outputs
    # out inside the timed region.
    e2e_ms = e2e_pipelined(fa, w, q, k, v, bufs, ws, drop, stream, device,
                           max(1, min(args.steps, args.e2e_steps)), world)
    sampler.stop()
    clocks = sampler.summary(t0, t1, fallback_window=(t_warm, t1))

    if rank != 0:
        return 0
    flops = step_flops(w)
    value = world * flops * args.steps * passes / (total_ms * 1e-3) / 1e12
    achieved = flops / (kern_ms_max * 1e-3) / 1e12
    peak, peak_sustained, peak_src = measured_peaks()
    peak_src = f"{peak_src} bf16 burst"
    dtype_check = None
    if w["dtype"] == "fp16":
        dtype_check = dtype_peak_check(device)
        peak_src += (" x the nominal fp16/bf16 dense ratio 1 (cuBLAS probe in this run: "
                     f"{dtype_check['fp16_over_bf16']:.3f})")
    traffic, traffic_note = stored_traffic(w["name"])
    io = io_bytes(w)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "timed_passes": passes,
        "ms_per_step": total_ms / (args.steps * passes), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": w["name"], "B": B, "H": H, "N": N, "d": d,
                   "causal": w["causal"], "seed": w["seed"], "scale": w["scale"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "entry": ("fa_fwd_dropout" if drop > 0 else
                             "fa_fwd_ws" if ws is not None else "fa_fwd"),
                   "dropout": drop,
                   "tail": (f"last-round units split along keys (workspace {ws_bytes / 2**20:.1f} MiB)"
                            if ws is not None else "whole units only"),
                   "l2": (f"{replicas} rotating input replicas "
                          f"({replicas * per_replica / 2**20:.0f} MiB"
                          f"{' > L2' if replicas * per_replica > L2_BYTES else ', < L2: launch-bound size'})")
                   if replicas > 1 else "inputs larger than L2"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": peak_src, "dtype_peak_check": dtype_check,
                     "frac_of_sustained": achieved / peak_sustained if peak_sustained else None,
                     "kernel_ms": kern_ms_max, "flops_per_launch": flops,
                     "traffic": traffic,
                     "traffic_note": traffic_note,
                     "traffic_scope": ("dram__bytes read + write during one launch; O lines still "
                                       "dirty in L2 when the kernel ends are written back after "
                                       "it, so with O smaller than L2 the figure can fall below "
                                       "the compulsory bytes"),
                     "compulsory_bytes": io["h2d"] + io["d2h"]},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": io["h2d"], "d2h_bytes_per_step": io["d2h"],
                "ms_per_step": e2e_ms, "steps": max(1, min(args.steps, args.e2e_steps)),
                "pipelining": ("consecutive steps overlapped over two device buffer sets: "
                               "q, k, v uploads on three streams, attention_forward on the "
                               "compute stream, downloads on a fifth")},
        "clocks": clocks,
        "gpu_launches": args.steps * passes,
        "gpu": torch.cuda.get_device_name(device),
    }
    if graph is not None:
        line["graph_replay"] = {"launches": 1000, "us_per_launch": graph * 1e3,
                                "tflops": flops / (graph * 1e-3) / 1e12,
                                "note": "100 launches captured in one CUDA graph, replayed 10 times"}
    if not args.no_cpu_baseline:
        if drop > 0:
            tf, dt, heads, cores, desc = dropout_oracle_sample(w, q, k, v, None, drop,
                                                               args.cpu_seconds)
        else:
            tf, dt, heads, cores, desc = oracle_sample(w, q, k, v, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    print(json.dumps(line), flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(json.dumps(line) + "\n")
    return 0


def run_ours_bwd(args, w):
    """The backward pass: one step = one fa_bwd call (two kernels) on
    inputs, the forward's O and LSE, and dO resident in device memory."""
    import exact_tiled_attention_14_gb300 as fa

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    fa.load_library()

    sampler = ClockSampler(local).start()
    q, k, v = seeded_inputs.make_workload_qkv(w)
    dout = seeded_inputs.make_dout(w["B"], w["H"], w["N"], w["d"], w["dtype"], seed=w["seed"])
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    io = io_bytes_bwd(w)
    per_replica = io["h2d"] + io["d2h"] + B * H * N * 4
    replicas = 1 if per_replica > 2 * L2_BYTES else int(math.ceil(2 * L2_BYTES / per_replica)) + 1
    replicas = min(replicas, 64)
    stream = torch.cuda.current_stream(device)
    code = fa.dtype_code(q.dtype)
    bufs = []
    drop = args.dropout
    for _ in range(replicas):
        dq_, dk_, dv_, do_ = (t.to(device) for t in (q, k, v, dout))
        if drop > 0:
            o, lse = fa.attention_forward_dropout(dq_, dk_, dv_, drop, w["seed"], 0,
                                                  causal=w["causal"], scale=w["scale"],
                                                  stream=stream)
        else:
            o, lse = fa.attention_forward(dq_, dk_, dv_, causal=w["causal"], scale=w["scale"],
                                          stream=stream)
        gq, gk, gv = torch.empty_like(dq_), torch.empty_like(dk_), torch.empty_like(dv_)
        delta = torch.empty((B, H, N), dtype=torch.float32, device=device)
        bufs.append((dq_, dk_, dv_, o, lse, do_, gq, gk, gv, delta))

    onepass = args.onepass
    ws_bytes = fa.fa_bwd_onepass_workspace_size(B, H, N, d) if onepass else 0
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device) if onepass else None
    entry = ("fa_bwd_onepass" if onepass else "fa_bwd") + ("_dropout" if drop > 0 else "")

    def step(i):
        if drop > 0 and onepass:
            rc = fa.fa_bwd_onepass_dropout(*bufs[i % replicas], B, H, N, d, w["causal"],
                                           w["scale"], drop, w["seed"], 0, code, ws, ws_bytes,
                                           stream)
        elif drop > 0:
            rc = fa.fa_bwd_dropout(*bufs[i % replicas], B, H, N, d, w["causal"], w["scale"], drop,
                                   w["seed"], 0, code, stream)
        elif onepass:
            rc = fa.fa_bwd_onepass(*bufs[i % replicas], B, H, N, d, w["causal"], w["scale"], code,
                                   ws, ws_bytes, stream)
        else:
            rc = fa.fa_bwd(*bufs[i % replicas], B, H, N, d, w["causal"], w["scale"], code, stream)
        if rc:
            raise fa.FaError(rc, entry)

    t_warm = time.time()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st, word = fa.fa_status(stream)
    if st:
        raise fa.FaError(st, f"warmup status {word:#x}")
    total_ms, per_step, passes, t0, t1 = timed_region(step, args.steps, args.min_timed_ms, stream,
                                                      world, device)
    kern_ms = max_over_ranks(statistics.mean(per_step), world, device)
    st, word = fa.fa_status(stream)
    if st:
        raise fa.FaError(st, f"timed status {word:#x}")

    # end to end: pinned host q, k, v, o, lse, dO in; dQ, dK, dV out
    hosts = [t.pin_memory() for t in (q, k, v)]
    dq_, dk_, dv_, o, lse, do_ = bufs[0][:6]
    ho, hl = o.cpu().pin_memory(), lse.cpu().pin_memory()
    hdo = dout.pin_memory()
    outs = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(3)]
    e2e_steps = max(1, min(args.steps, args.e2e_steps))

    def e2e_step():
        for dst, src in zip((dq_, dk_, dv_, o, lse, do_), hosts + [ho, hl, hdo]):
            dst.copy_(src, non_blocking=True)
        if onepass:
            grads = fa.attention_backward_onepass(dq_, dk_, dv_, o, lse, do_, causal=w["causal"],
                                                  scale=w["scale"], workspace=ws, stream=stream,
                                                  dropout_p=drop, seed=w["seed"], offset=0)
        elif drop > 0:
            grads = fa.attention_backward_dropout(dq_, dk_, dv_, o, lse, do_, drop, w["seed"], 0,
                                                  causal=w["causal"], scale=w["scale"],
                                                  stream=stream)
        else:
            grads = fa.attention_backward(dq_, dk_, dv_, o, lse, do_, causal=w["causal"],
                                          scale=w["scale"], stream=stream)
        for dst, src in zip(outs, grads):
            dst.copy_(src, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, device)
    sampler.stop()
    clocks = sampler.summary(t0, t1, fallback_window=(t_warm, t1))

    if rank != 0:
        return 0
    flops = step_flops_bwd(w)
    value = world * flops * args.steps * passes / (total_ms * 1e-3) / 1e12
    achieved = flops / (kern_ms * 1e-3) / 1e12
    peak, peak_sustained, peak_src = measured_peaks()
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "timed_passes": passes,
        "ms_per_step": total_ms / (args.steps * passes), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": w["name"], "pass": "backward", "B": B, "H": H, "N": N, "d": d,
                   "causal": w["causal"], "seed": w["seed"], "scale": w["scale"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "entry": entry, "dropout": drop,
                   "l2": (f"{replicas} rotating replicas ({replicas * per_replica / 2**20:.0f} MiB)"
                          if replicas > 1 else "inputs larger than L2")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} bf16 burst",
                     "frac_of_sustained": achieved / peak_sustained if peak_sustained else None,
                     "kernel_ms": kern_ms, "flops_per_launch": flops,
                     "scope": (f"one {entry} call: D, one-pass and dQ conversion kernels together"
                               if onepass else
                               f"one {entry} call: D, dK/dV and dQ kernels together"),
                     "traffic": None, "traffic_note": "no ncu DRAM capture of the backward yet"},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": io["h2d"], "d2h_bytes_per_step": io["d2h"],
                "ms_per_step": e2e_ms, "steps": e2e_steps},
        "clocks": clocks,
        # the D pass and the dK/dV + dQ grid (one-pass: also the dQ conversion;
        # the workspace clearing is a cudaMemsetAsync)
        "gpu_launches": (3 if onepass else 2) * args.steps * passes,
        "gpu": torch.cuda.get_device_name(device),
    }
    if not args.no_cpu_baseline:
        if drop > 0:
            tf, dt, heads, cores, desc = dropout_oracle_sample(w, q, k, v, dout, drop,
                                                               args.cpu_seconds)
        else:
            tf, dt, heads, cores, desc = oracle_grad_sample(w, q, k, v, dout, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    print(json.dumps(line), flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(json.dumps(line) + "\n")
    return 0


def run_ours_decode(args, w):
    """Split-KV decoding: one step = one fa_decode call (partial and combine
    kernels) of the workload's queries against its cache, resident in device
    memory.  HBM-bound: the metric is the K/V bytes read per second."""
    import exact_tiled_attention_14_gb300 as fa

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    fa.load_library()
    sampler = ClockSampler(local).start()
    B, H, Nq, Nk, d = w["B"], w["H"], w["Nq"], w["Nk"], w["d"]
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, w["dtype"], seed=w["seed"])
    kv_bytes = 2 * B * H * Nk * d * 2
    io = dict(h2d=B * H * Nq * d * 2 + kv_bytes, d2h=B * H * Nq * (d * 2 + 4))
    per_replica = io["h2d"] + io["d2h"]
    replicas = 1 if per_replica > 2 * L2_BYTES else int(math.ceil(2 * L2_BYTES / per_replica)) + 1
    replicas = min(replicas, 64)
    stream = torch.cuda.current_stream(device)
    code = fa.dtype_code(q.dtype)
    ws_bytes = fa.fa_decode_workspace_size(B, H, Nq, Nk, d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)
    bufs = []
    for _ in range(replicas):
        dq_, dk_, dv_ = (t.to(device) for t in (q, k, v))
        bufs.append((dq_, dk_, dv_, torch.empty_like(dq_),
                     torch.empty((B, H, Nq), dtype=torch.float32, device=device)))

    def step(i):
        dq_, dk_, dv_, o, lse = bufs[i % replicas]
        rc = fa.fa_decode(dq_, dk_, dv_, o, lse, B, H, Nq, Nk, d, w["causal"], w["scale"], code,
                          ws, ws_bytes, stream)
        if rc:
            raise fa.FaError(rc, "fa_decode")

    t_warm = time.time()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st, word = fa.fa_status(stream)
    if st:
        raise fa.FaError(st, f"warmup status {word:#x}")
    total_ms, per_step, passes, t0, t1 = timed_region(step, args.steps, args.min_timed_ms, stream,
                                                      world, device)
    kern_ms = max_over_ranks(statistics.mean(per_step), world, device)
    st, word = fa.fa_status(stream)
    if st:
        raise fa.FaError(st, f"timed status {word:#x}")

    # end to end: pinned host q and cache in, o and lse out
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hl = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    dq_, dk_, dv_, o, lse = bufs[0]
    e2e_steps = max(1, min(args.steps, args.e2e_steps))

    def e2e_step():
        dq_.copy_(hq, non_blocking=True)
        dk_.copy_(hk, non_blocking=True)
        dv_.copy_(hv, non_blocking=True)
        fa.attention_decode(dq_, dk_, dv_, causal=w["causal"], scale=w["scale"], out=o, lse=lse,
                            workspace=ws, stream=stream)
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, device)
    sampler.stop()
    clocks = sampler.summary(t0, t1, fallback_window=(t_warm, t1))
    if rank != 0:
        return 0
    gbs = lambda ms: world * kv_bytes / (ms * 1e-3) / 1e9   # noqa: E731
    peak, src = measured_hbm()
    line = {
        "metric": METRIC_DEC, "value": world * kv_bytes * args.steps * passes / (total_ms * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "timed_passes": passes,
        "ms_per_step": total_ms / (args.steps * passes), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": w["name"], "pass": "decode", "B": B, "H": H, "Nq": Nq, "Nk": Nk,
                   "d": d, "causal": w["causal"], "seed": w["seed"], "scale": w["scale"],
                   "entry": "fa_decode", "parallelism": "single GPU" if world == 1 else f"replicas x{world}",
                   "l2": (f"{replicas} rotating replicas ({replicas * per_replica / 2**20:.0f} MiB)"
                          if replicas > 1 else "cache larger than L2")},
        "roofline": {"bound": "hbm", "achieved": gbs(kern_ms), "peak": peak, "unit": "GB/s",
                     "frac": gbs(kern_ms) / peak, "peak_source": src, "kernel_ms": kern_ms,
                     "bytes_per_launch": kv_bytes,
                     "scope": "one fa_decode call: split-KV partial and combine kernels",
                     "traffic": None, "traffic_note": "no ncu DRAM capture of the decode kernels yet"},
        "e2e": {"value": gbs(e2e_ms), "unit": "GB/s", "h2d_bytes_per_step": io["h2d"],
                "d2h_bytes_per_step": io["d2h"], "ms_per_step": e2e_ms, "steps": e2e_steps},
        "clocks": clocks,
        "gpu_launches": 2 * args.steps * passes,
        "gpu": torch.cuda.get_device_name(device),
    }
    print(json.dumps(line), flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(json.dumps(line) + "\n")
    return 0


def kv_oracle_sample(w, q, k, v, seqlens, budget_s, start_head=0):
    """Time the float64 oracle on whole (batch, head) pairs of an fa_fwd_kv
    workload for about budget_s: each row at its absolute position against
    the batch's keys.  Returns (TFLOP/s, seconds, heads, cores, description)."""
    import numpy as np
    import oracle
    lib = oracle.load()
    B, H = w["B"], w["H"]
    pos = kv_positions(w, seqlens)
    cores = oracle.num_threads(lib)
    done, spent, flops = 0, 0.0, 0.0
    while done < B * H and (done == 0 or spent < budget_s):
        b, h = divmod((start_head + done) % (B * H), H)
        n, off = pos[b]
        rows = np.arange(w["Nq"], dtype=np.int64) + off
        qh = q[b, h].double().numpy()
        kh, vh = (t[b, h, :n].double().numpy() for t in (k, v))
        t0 = time.perf_counter()
        oracle.attention_rows(qh, rows, kh, vh, causal=bool(w["causal"]), scale=w["scale"], lib=lib)
        spent += time.perf_counter() - t0
        flops += 4.0 * w["d"] * kv_visible_pairs(w, n, off)
        done += 1
    desc = (f"{done} of {B * H} whole (batch, head) pairs of {w['name']} (float64, {cores} "
            "threads); FLOPs counted per pair from its visible keys")
    return flops / spent / 1e12, spent, done, cores, desc


def run_ours_kv(args, w):
    """Queries against a key set of another length: one step = one fa_fwd_kv
    launch over the workload resident in device memory (key counts included)."""
    import exact_tiled_attention_14_gb300 as fa

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    fa.load_library()
    sampler = ClockSampler(local).start()
    B, H, Nq, Nk, d = w["B"], w["H"], w["Nq"], w["Nk"], w["d"]
    q, k, v = seeded_inputs.make_decode(B, H, Nq, Nk, d, w["dtype"], seed=w["seed"])
    seqlens = seeded_inputs.make_seqlens(B, Nk, w["seed"]) if w["padded"] else None
    mode = fa.CAUSAL_MODES[w["causal"]]
    flops = step_flops_kv(w, seqlens)
    io = dict(h2d=B * H * (Nq + 2 * Nk) * d * 2 + (0 if seqlens is None else 4 * B),
              d2h=B * H * Nq * (d * 2 + 4))
    per_replica = io["h2d"] + io["d2h"]
    replicas = 1 if per_replica > 2 * L2_BYTES else int(math.ceil(2 * L2_BYTES / per_replica)) + 1
    replicas = min(replicas, 64)
    stream = torch.cuda.current_stream(device)
    code = fa.dtype_code(q.dtype)
    dsl = None if seqlens is None else seqlens.to(device)
    bufs = []
    for _ in range(replicas):
        dq_, dk_, dv_ = (t.to(device) for t in (q, k, v))
        bufs.append((dq_, dk_, dv_, torch.empty_like(dq_),
                     torch.empty((B, H, Nq), dtype=torch.float32, device=device)))

    def step(i):
        dq_, dk_, dv_, o, lse = bufs[i % replicas]
        rc = fa.fa_fwd_kv(dq_, dk_, dv_, o, lse, B, H, Nq, Nk, d, d, mode, dsl, w["scale"],
                          code, stream)
        if rc:
            raise fa.FaError(rc, "fa_fwd_kv")

    t_warm = time.time()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st, word = fa.fa_status(stream)
    if st:
        raise fa.FaError(st, f"warmup status {word:#x}")
    total_ms, per_step, passes, t0, t1 = timed_region(step, args.steps, args.min_timed_ms, stream,
                                                      world, device)
    kern_ms = max_over_ranks(statistics.mean(per_step), world, device)
    st, word = fa.fa_status(stream)
    if st:
        raise fa.FaError(st, f"timed status {word:#x}")

    # end to end: pinned host q, k, v (and key counts) in, o and lse out
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    hsl = None if seqlens is None else seqlens.pin_memory()
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hl = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    dq_, dk_, dv_, o, lse = bufs[0]
    e2e_steps = max(1, min(args.steps, args.e2e_steps))

    def e2e_step():
        dq_.copy_(hq, non_blocking=True)
        dk_.copy_(hk, non_blocking=True)
        dv_.copy_(hv, non_blocking=True)
        if hsl is not None:
            dsl.copy_(hsl, non_blocking=True)
        fa.attention_forward_kv(dq_, dk_, dv_, causal=w["causal"], seqlens_k=dsl,
                                scale=w["scale"], out=o, lse=lse, stream=stream)
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, device)
    # the backward pass of the same workload (fa_bwd_kv; value width = d)
    dout = seeded_inputs.make_dout(B, H, Nq, d, w["dtype"], seed=w["seed"]).to(device)
    o_f, l_f = fa.attention_forward_kv(dq_, dk_, dv_, causal=w["causal"], seqlens_k=dsl,
                                       scale=w["scale"])
    bwd_ms = time_launches(lambda: fa.attention_backward_kv(
        dq_, dk_, dv_, o_f, l_f, dout, causal=w["causal"], seqlens_k=dsl, scale=w["scale"]),
        max(5, args.steps // 4))
    sampler.stop()
    clocks = sampler.summary(t0, t1, fallback_window=(t_warm, t1))
    if rank != 0:
        return 0
    achieved = flops / (kern_ms * 1e-3) / 1e12
    peak, peak_sustained, peak_src = measured_peaks()
    traffic, traffic_note = stored_traffic(w["name"])
    line = {
        "metric": METRIC_KV, "value": world * flops * args.steps * passes / (total_ms * 1e-3) / 1e12,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "timed_passes": passes,
        "ms_per_step": total_ms / (args.steps * passes), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": w["name"], "pass": "kv", "B": B, "H": H, "Nq": Nq, "Nk": Nk,
                   "d": d, "causal": w["causal"], "seed": w["seed"], "scale": w["scale"],
                   "seqlens_k": None if seqlens is None else seqlens.tolist(),
                   "entry": "fa_fwd_kv",
                   "parallelism": "single GPU" if world == 1 else f"replicas x{world}",
                   "l2": (f"{replicas} rotating replicas ({replicas * per_replica / 2**20:.0f} MiB)"
                          if replicas > 1 else "inputs larger than L2")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} bf16 burst",
                     "frac_of_sustained": achieved / peak_sustained if peak_sustained else None,
                     "kernel_ms": kern_ms, "flops_per_launch": flops,
                     "traffic": traffic, "traffic_note": traffic_note,
                     "compulsory_bytes": io["h2d"] + io["d2h"]},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": io["h2d"], "d2h_bytes_per_step": io["d2h"],
                "ms_per_step": e2e_ms, "steps": e2e_steps},
        "clocks": clocks,
        "gpu_launches": args.steps * passes,
        "gpu": torch.cuda.get_device_name(device),
        "backward": backward_line(bwd_ms, flops, "fa_bwd_kv", peak),
    }
    if not args.no_cpu_baseline:
        tf, dt, heads, cores, desc = kv_oracle_sample(w, q, k, v, seqlens, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    print(json.dumps(line), flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(json.dumps(line) + "\n")
    return 0


def run_ours_varlen(args, w):
    """Packed variable-length batch: one step = one fa_fwd_varlen launch over
    the packed workload resident in device memory.  For context the same
    batch padded to its longest sequence is also timed through fa_fwd_kv
    (key counts given, padded query rows still computed)."""
    import exact_tiled_attention_14_gb300 as fa

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    fa.load_library()
    sampler = ClockSampler(local).start()
    B, H, d = w["B"], w["H"], w["d"]
    lens = seeded_inputs.varlen_lengths(B, w["lo"], w["hi"], w["seed"])
    q, k, v, cu_q, cu_k = seeded_inputs.make_varlen(lens, lens, H, d, w["dtype"], seed=w["seed"])
    total, max_len = sum(lens), max(lens)
    mode = fa.CAUSAL_MODES[w["causal"]]
    flops = sum(4.0 * d * H * kv_visible_pairs(dict(Nq=n, causal=w["causal"]), n, 0)
                for n in lens)
    io = dict(h2d=3 * total * H * d * 2 + 2 * 4 * (B + 1), d2h=total * H * (d * 2 + 4))
    stream = torch.cuda.current_stream(device)
    code = fa.dtype_code(q.dtype)
    per_replica = io["h2d"] + io["d2h"]
    replicas = 1 if per_replica > 2 * L2_BYTES else int(math.ceil(2 * L2_BYTES / per_replica)) + 1
    replicas = min(replicas, 64)
    dcq, dck = cu_q.to(device), cu_k.to(device)
    bufs = []
    for _ in range(replicas):
        dq_, dk_, dv_ = (t.to(device) for t in (q, k, v))
        bufs.append((dq_, dk_, dv_, torch.empty_like(dq_),
                     torch.empty((H, total), dtype=torch.float32, device=device)))

    def step(i):
        dq_, dk_, dv_, o, lse = bufs[i % replicas]
        rc = fa.fa_fwd_varlen(dq_, dk_, dv_, o, lse, dcq, dck, B, H, max_len, total, total, d, d,
                              mode, w["scale"], code, stream)
        if rc:
            raise fa.FaError(rc, "fa_fwd_varlen")

    def timed(fn, steps):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        st, word = fa.fa_status(stream)
        if st:
            raise fa.FaError(st, f"warmup status {word:#x}")
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier(world, device)
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(steps):
            starts[i].record(stream)
            fn(i)
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier(world, device)
        t1 = time.time()
        st, word = fa.fa_status(stream)
        if st:
            raise fa.FaError(st, f"timed status {word:#x}")
        total_ms = max_over_ranks(starts[0].elapsed_time(ends[-1]), world, device)
        kern_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends)),
                                 world, device)
        return total_ms, kern_ms, t0, t1

    t_warm = time.time()
    total_ms, kern_ms, t0, t1 = timed(step, args.steps)
    clocks_window = (t0, t1)

    # end to end: pinned host packed q, k, v and offsets in, o and lse out
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    hcq, hck = cu_q.pin_memory(), cu_k.pin_memory()
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hl = torch.empty((H, total), dtype=torch.float32).pin_memory()
    dq_, dk_, dv_, o, lse = bufs[0]
    e2e_steps = max(1, min(args.steps, args.e2e_steps))

    def e2e_step():
        dq_.copy_(hq, non_blocking=True)
        dk_.copy_(hk, non_blocking=True)
        dv_.copy_(hv, non_blocking=True)
        dcq.copy_(hcq, non_blocking=True)
        dck.copy_(hck, non_blocking=True)
        fa.attention_forward_varlen(dq_, dk_, dv_, dcq, dck, max_len, causal=w["causal"],
                                    scale=w["scale"], out=o, lse=lse, stream=stream)
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, device)

    # the backward pass of the same batch (fa_bwd_varlen)
    dout = torch.randn(q.shape, generator=torch.Generator("cpu").manual_seed(w["seed"]))
    dout = dout.to(q.dtype).to(device)
    o_f, l_f = fa.attention_forward_varlen(dq_, dk_, dv_, dcq, dck, max_len, causal=w["causal"],
                                           scale=w["scale"])
    bwd_ms = time_launches(lambda: fa.attention_backward_varlen(
        dq_, dk_, dv_, o_f, l_f, dout, dcq, dck, max_len, max_len, causal=w["causal"],
        scale=w["scale"]), max(5, args.steps // 4))
    del dout, o_f, l_f

    # the same batch padded to the longest sequence, through fa_fwd_kv
    del bufs
    pq = torch.zeros((B, H, max_len, d), dtype=q.dtype, device=device)
    pk, pv = torch.zeros_like(pq), torch.zeros_like(pq)
    for b, n in enumerate(lens):
        a = int(cu_q[b])
        pq[b, :, :n] = q[a:a + n].to(device).transpose(0, 1)
        pk[b, :, :n] = k[a:a + n].to(device).transpose(0, 1)
        pv[b, :, :n] = v[a:a + n].to(device).transpose(0, 1)
    po = torch.empty_like(pq)
    pl = torch.empty((B, H, max_len), dtype=torch.float32, device=device)
    psl = torch.tensor(lens, dtype=torch.int32, device=device)

    def padded_step(i):
        rc = fa.fa_fwd_kv(pq, pk, pv, po, pl, B, H, max_len, max_len, d, d, mode, psl,
                          w["scale"], code, stream)
        if rc:
            raise fa.FaError(rc, "fa_fwd_kv (padded)")

    _, padded_ms, _, _ = timed(padded_step, max(10, args.steps // 4))
    sampler.stop()
    clocks = sampler.summary(*clocks_window, fallback_window=(t_warm, clocks_window[1]))
    if rank != 0:
        return 0
    achieved = flops / (kern_ms * 1e-3) / 1e12
    peak, peak_sustained, peak_src = measured_peaks()
    traffic, traffic_note = stored_traffic(w["name"])
    line = {
        "metric": METRIC_VARLEN, "value": world * flops * args.steps / (total_ms * 1e-3) / 1e12,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": w["name"], "pass": "varlen", "B": B, "H": H, "d": d,
                   "causal": w["causal"], "seed": w["seed"], "scale": w["scale"],
                   "lengths": lens, "total_tokens": total, "entry": "fa_fwd_varlen",
                   "padded_equivalent": {"entry": "fa_fwd_kv", "ms": padded_ms,
                                         "note": "same batch padded to the longest sequence"},
                   "parallelism": "single GPU" if world == 1 else f"replicas x{world}",
                   "l2": (f"{replicas} rotating replicas ({replicas * per_replica / 2**20:.0f} MiB)"
                          if replicas > 1 else "inputs larger than L2")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} bf16 burst",
                     "frac_of_sustained": achieved / peak_sustained if peak_sustained else None,
                     "kernel_ms": kern_ms, "flops_per_launch": flops,
                     "traffic": traffic, "traffic_note": traffic_note,
                     "compulsory_bytes": io["h2d"] + io["d2h"]},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": io["h2d"], "d2h_bytes_per_step": io["d2h"],
                "ms_per_step": e2e_ms, "steps": e2e_steps},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "gpu": torch.cuda.get_device_name(device),
        "backward": backward_line(bwd_ms, flops, "fa_bwd_varlen", peak),
    }
    if not args.no_cpu_baseline:
        import numpy as np
        import oracle
        lib = oracle.load()
        cores = oracle.num_threads(lib)
        spent, done_flops, heads = 0.0, 0.0, 0
        order = sorted(range(B), key=lambda b: lens[b])       # shortest sequences first
        for b in order:
            n, a = lens[b], int(cu_q[b])
            for h in range(H):
                t_a = time.perf_counter()
                oracle.attention_rows(q[a:a + n, h].double().numpy(), np.arange(n, dtype=np.int64),
                                      k[a:a + n, h].double().numpy(), v[a:a + n, h].double().numpy(),
                                      causal=True, scale=w["scale"], lib=lib)
                spent += time.perf_counter() - t_a
                done_flops += 4.0 * d * kv_visible_pairs(dict(Nq=n, causal=w["causal"]), n, 0)
                heads += 1
                if spent >= args.cpu_seconds:
                    break
            if spent >= args.cpu_seconds:
                break
        line["cpu_baseline"] = {"value": done_flops / spent / 1e12, "unit": "TFLOP/s",
                                "cores": cores, "kind": "oracle", "seconds": spent,
                                "sample": f"{heads} whole (sequence, head) pairs of {w['name']}, "
                                          "shortest sequences first (float64)"}
    print(json.dumps(line), flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(json.dumps(line) + "\n")
    return 0


def measured_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(path))["hbm_gbs"]), "measured HBM copy"
    except (OSError, ValueError, KeyError, TypeError):
        return 6800.0, "fallback"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--min-timed-ms", type=float, default=1000.0,
                    help="repeat the --steps pass until this much device time is timed")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="one of: " + ", ".join(x["name"] for x in seeded_inputs.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None,
                    help="override B of the workload (smaller profiling captures)")
    ap.add_argument("--heads", type=int, default=None, help="override H of the workload")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--split", action="store_true",
                    help="time fa_fwd_ws (last round split along keys) instead of fa_fwd")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="dropout probability on the attention weights (fa_fwd_dropout, or "
                         "fa_bwd_dropout with --pass bwd); 0 = none")
    ap.add_argument("--onepass", action="store_true",
                    help="with --pass bwd: time fa_bwd_onepass (fa_bwd_onepass_dropout with "
                         "--dropout) instead of fa_bwd")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "decode", "kv", "varlen"], default="fwd",
                    help="time the forward pass (default), the backward pass (fa_bwd), "
                         "split-KV decoding (fa_decode; --workload names a decoding workload) "
                         ", fa_fwd_kv (--workload names a kv workload) or fa_fwd_varlen")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.pass_ == "decode":
        name = args.workload if args.workload != DEFAULT_WORKLOAD else \
            seeded_inputs.DECODE_WORKLOADS[-1]["name"]
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the decoding pass has no reference arm; the oracle checks it in tests"}))
            return 0
        wd = seeded_inputs.decode_workload(name)
        if args.batch is not None or args.heads is not None:
            wd["B"] = args.batch if args.batch is not None else wd["B"]
            wd["H"] = args.heads if args.heads is not None else wd["H"]
            wd["name"] = f"{wd['name']}@B{wd['B']}H{wd['H']}"
        return run_ours_decode(args, wd)
    if args.pass_ == "varlen":
        name = args.workload if args.workload != DEFAULT_WORKLOAD else \
            seeded_inputs.VARLEN_WORKLOADS[0]["name"]
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the varlen pass has no reference arm; the oracle checks it in tests "
                              "and its cpu_baseline times it"}))
            return 0
        return run_ours_varlen(args, seeded_inputs.varlen_workload(name))
    if args.pass_ == "kv":
        name = args.workload if args.workload != DEFAULT_WORKLOAD else \
            seeded_inputs.KV_WORKLOADS[0]["name"]
        wk = seeded_inputs.kv_workload(name)
        if args.batch is not None or args.heads is not None:
            wk["B"] = args.batch if args.batch is not None else wk["B"]
            wk["H"] = args.heads if args.heads is not None else wk["H"]
            wk["name"] = f"{wk['name']}@B{wk['B']}H{wk['H']}"
        if args.impl == "reference":
            return run_reference_kv(args, wk)
        return run_ours_kv(args, wk)
    w = seeded_inputs.workload(args.workload)
    if args.batch is not None or args.heads is not None:
        w["B"] = args.batch if args.batch is not None else w["B"]
        w["H"] = args.heads if args.heads is not None else w["H"]
        w["name"] = f"{w['name']}@B{w['B']}H{w['H']}"
    if args.impl == "reference":
        return run_reference(args, w)
    if args.pass_ == "bwd":
        return run_ours_bwd(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
