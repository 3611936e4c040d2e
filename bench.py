"""Benchmark of the attention forward: TFLOP/s on the d=128, S=4096 workload.

One step = one forward over the whole batch in each masking mode: a full
(non-causal) launch and a causal launch on the same seeded inputs
(B=2, H=32, S_q=S_k=4096, d=128, bf16, scale=1/sqrt(128); Q, K ~ N(0,1),
V ~ U(-1,1)).  FLOPs per step = 4·B·H·S²·d (full) + half of that (causal).

Prints one JSON line (rank 0).  ``value`` is device-timed throughput with
inputs resident in HBM; ``e2e`` is the same metric through the host-buffer C
entry point, copies included; ``roofline`` is for the dominant launch (the
full one); ``cpu_baseline`` times the fp64 oracle on a bounded sample;
``splitkv`` reports the split-KV forward on the decode workload (one query row
per head against 32768 keys) in HBM GB/s, and ``backward`` the backward pass
(dQ, dK, dV) on the same c3 inputs in TFLOP/s; both are measured after the
timed steps and are not part of ``value``.

``--impl reference`` times the fp64 CPU oracle instead (there is no runnable
reference implementation: the attention page is Rust that emits PTX for
sm_90, with its kernel body absent).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "c3"
METRIC = "attention fwd TFLOP/s (bf16, causal & non-causal) and % of GB300 dense peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 - 0.25 <= s[0] <= t1 + 0.25] or self.samples
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i, v in enumerate(s[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[1] for s in win),
                "sm_max_mhz": max(s[2] for s in win), "reasons": reasons, "samples": len(win)}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest `value` over all ranks (the job time is the slowest rank's)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s when every rank runs its own replica of the workload."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


# Source files that make up each profiled kernel: a DRAM-traffic figure is
# used only while these files are byte-identical to the ones it was taken on.
FWD_SOURCES = ("attn_fwd.cuh", "attn_inst.cu", "attn_launch.h", "sm100.cuh")
BWD_SOURCES = ("attn_bwd.cuh", "attn_bwd_wide.cuh", "attn_bwd_inst.cu", "attn_launch.h", "sm100.cuh")
KERNEL_SOURCES = {
    "attn_fwd_d128_bf16_full_c3": FWD_SOURCES,
    "attn_fwd_d128_bf16_causal_c3": FWD_SOURCES,
    "attn_fwd_splitkv_d128_bf16_decode": FWD_SOURCES + ("attn_combine.cu",),
    "attn_bwd_d128_bf16_full_c3": BWD_SOURCES,
    "attn_bwd_d128_bf16_causal_c3": BWD_SOURCES,
}


def kernel_source_digest(names) -> str:
    """sha256 over the named kernel sources; ties recorded DRAM traffic to the code it was taken on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_53_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def measured_traffic(key: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not isinstance(rec, dict) or rec.get("sources_sha256") != kernel_source_digest(KERNEL_SOURCES[key]):
        return None
    return rec.get("bytes")


def cpu_baseline(budget_s: float = 12.0):
    """The fp64 oracle, as it stands, on whole heads of the workload until the budget is spent."""
    import numpy as np  # noqa: F401

    import oracle
    from exact_attention_53_gb300.workloads import WORKLOADS, workload_qkv

    w = WORKLOADS[WORKLOAD]
    q, k, v = workload_qkv(w)
    flops = 0.0
    heads = 0
    t0 = time.perf_counter()
    while True:
        b, h = divmod(heads % (w.B * w.H), w.H)
        causal = heads % 2 == 1
        oracle.attention_forward(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                 causal=causal, scale=w.scale)
        flops += 4.0 * w.S_q * w.S_k * w.d / (2 if causal else 1)
        heads += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{heads} whole (b,h) heads of {WORKLOAD} (B=2,H=32,S=4096,d=128), "
                      f"alternating full/causal, fp64 numpy, {dt:.1f} s"}


def cpu_per_config():
    """The fp64 oracle timed on a bounded sample of every workload (wall clock, host cores):
    c1 and c2 whole heads; c4 and c5 a block of 512 query rows from the middle of one head
    (FLOPs counted exactly: a causal row i sees i + 1 keys)."""
    import numpy as np

    import oracle
    from exact_attention_53_gb300.workloads import WORKLOADS, workload_qkv

    out = {}
    for name in ("c1", "c2", "c4", "c5"):
        w = WORKLOADS[name]
        causal = w.causal[0]
        q, k, v = workload_qkv(w)
        if name in ("c1", "c2"):
            rows = np.arange(w.S_q)
            what = "one whole (b,h) head"
        else:
            rows = np.arange(w.S_q // 2 - 256, w.S_q // 2 + 256)
            what = f"rows {rows[0]}..{rows[-1]} of one (b,h) head"
        keys = (rows + 1) if causal else np.full(rows.shape, w.S_k)
        flops = float(4 * w.d * keys.sum())
        t0 = time.perf_counter()
        oracle.attention_rows(q[0, 0], k[0, 0], v[0, 0], rows, causal=causal, scale=w.scale)
        dt = time.perf_counter() - t0
        out[name] = {"tflops": flops / dt / 1e12, "seconds": dt, "sample": what}
    return out


def measure_long(dev, stream, launches: int = 30):
    """The long-sequence workloads c4 (S = 16384, causal) and c5 (d = 256): median, p10 and p90
    of `launches` CUDA-event-timed launches after 10 warm-ups; inputs (≥ 201 MB) exceed L2."""
    import torch

    from exact_attention_53_gb300 import attn_fwd
    from exact_attention_53_gb300.binding import ATTN_DTYPE_BF16
    from exact_attention_53_gb300.workloads import WORKLOADS, workload_qkv

    peak = load_peaks()[0].get("bf16_tflops")
    out = {}
    for name in ("c4", "c5"):
        w = WORKLOADS[name]
        causal = w.causal[0]
        q, k, v = (t.to(dev) for t in workload_qkv(w))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S_q), dtype=torch.float32, device=dev)

        def launch():
            attn_fwd(q, k, v, o, lse, w.B, w.H, w.S_q, w.S_k, w.d, int(causal), w.scale,
                     ATTN_DTYPE_BF16, stream)

        for _ in range(10):
            launch()
        torch.cuda.synchronize(dev)
        ms = []
        for _ in range(launches):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch()
            b.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(a.elapsed_time(b))
        pc = percentiles(ms)
        tf = w.flops(causal) / (pc["median_ms"] * 1e-3) / 1e12
        out[name] = {"workload": f"{name}: B={w.B} H={w.H} S={w.S_q} d={w.d} {w.dtype} "
                                 f"{'causal' if causal else 'full'}",
                     **pc, "tflops": tf, "frac_of_peak": tf / peak if peak else None}
        del q, k, v, o, lse
    return out


def run_reference(args, rank, world):
    """The fp64 oracle on the host cores, K timed steps of one head pair each."""
    if rank != 0:
        return
    import oracle
    from exact_attention_53_gb300.workloads import WORKLOADS, workload_qkv

    w = WORKLOADS[WORKLOAD]
    q, k, v = workload_qkv(w)

    def step(i):
        b, h = divmod(i % (w.B * w.H), w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        for causal in (False, True):
            oracle.attention_forward(q[sl], k[sl], v[sl], causal=causal, scale=w.scale)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    flops_step = 4.0 * w.S_q * w.S_k * w.d * 1.5
    value = flops_step * args.steps / dt / 1e12
    sample = f"per step one (b,h) head of {WORKLOAD}, full + causal, fp64 numpy oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: one head per step of B=2,H=32,S_q=S_k=4096,d=128"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def measure_splitkv(dev, stream, iters: int = 50):
    """Split-KV forward on the decode workload: HBM GB/s, beside the one-pass kernel on it.

    Algorithmic bytes per call = Q, K, V read once + O and LSE written once
    (the partial results in the workspace are not counted).  K+V = 537 MB,
    larger than L2, so no flush is needed between calls.
    """
    import torch

    from exact_attention_53_gb300 import attn_fwd, attn_fwd_splitkv, attn_fwd_splitkv_plan
    from exact_attention_53_gb300.binding import ATTN_DTYPE_BF16
    from exact_attention_53_gb300.workloads import WORKLOADS, workload_qkv

    w = WORKLOADS["decode"]
    B, H, S_q, S_k, d = w.B, w.H, w.S_q, w.S_k, w.d
    q, k, v = (t.to(dev) for t in workload_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S_q), dtype=torch.float32, device=dev)
    n_split, ws = attn_fwd_splitkv_plan(B, H, S_q, S_k, d, ATTN_DTYPE_BF16, 0)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)

    def split():
        attn_fwd_splitkv(q, k, v, o, lse, B, H, S_q, S_k, d, w.scale, ATTN_DTYPE_BF16, 0, work,
                         ws, stream)

    def one_pass():
        attn_fwd(q, k, v, o, lse, B, H, S_q, S_k, d, 0, w.scale, ATTN_DTYPE_BF16, stream)

    def timed(fn, n):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    split_ms = timed(split, iters)
    one_ms = timed(one_pass, max(10, iters // 5))
    by = w.io_bytes()
    return {"workload": f"decode: B={B} H={H} S_q={S_q} S_k={S_k} d={d} bf16, full attention, "
                        f"Q,K,V~N(0,1)",
            "n_split": n_split, "workspace_bytes": ws, "bytes_per_call": by,
            "ms": split_ms, "gbs": by / (split_ms * 1e-3) / 1e9,
            "one_pass_ms": one_ms, "speedup_vs_one_pass": one_ms / split_ms,
            "gpu_launches_per_call": 2 if n_split > 1 else 1, "calls_timed": iters}


def percentiles(ms):
    """median, p10 and p90 of a list of launch times (ms)."""
    xs = sorted(ms)
    pick = lambda f: xs[min(len(xs) - 1, int(round(f * (len(xs) - 1))))]  # noqa: E731
    return {"median_ms": pick(0.5), "p10_ms": pick(0.1), "p90_ms": pick(0.9)}


def measure_short(dev, stream, launches: int = 50, graph_launches: int = 20, replays: int = 10):
    """The short-sequence workloads: c1 (one 128×128 tile; launch/latency-bound, so µs and
    GB/s of its 66 KB are reported, with a 256 MB L2 flush before every launch) and c2
    (S = 1024, d = 64, causal): median of `launches` CUDA-event-timed calls, each call's host
    work (validation, tensor maps, launch) inside its events.  Beside it, the device time
    alone: `graph_launches` calls captured back to back in one CUDA graph, replayed
    `replays` times, total ÷ launches (no host work and no L2 flush between them), and the
    host time of one call (wall clock over 200 calls, Python binding included)."""
    import time

    import torch

    from exact_attention_53_gb300 import attn_fwd
    from exact_attention_53_gb300.binding import ATTN_DTYPE_BF16, ATTN_DTYPE_F16
    from exact_attention_53_gb300.workloads import WORKLOADS, workload_qkv

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for name in ("c1", "c2"):
        w = WORKLOADS[name]
        q, k, v = (t.to(dev) for t in workload_qkv(w))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S_q), dtype=torch.float32, device=dev)
        causal = w.causal[0]
        code = ATTN_DTYPE_BF16 if w.dtype == "bf16" else ATTN_DTYPE_F16

        def launch():
            attn_fwd(q, k, v, o, lse, w.B, w.H, w.S_q, w.S_k, w.d, int(causal), w.scale, code,
                     stream)

        for _ in range(10):
            launch()
        torch.cuda.synchronize(dev)
        ms = []
        for _ in range(launches):
            if name == "c1":
                flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launch()
            b.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(a.elapsed_time(b))
        pc = percentiles(ms)
        t = pc["median_ms"] * 1e-3
        # device time: back-to-back launches replayed from a CUDA graph
        cap = torch.cuda.Stream(device=dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(graph_launches):
                attn_fwd(q, k, v, o, lse, w.B, w.H, w.S_q, w.S_k, w.d, int(causal), w.scale,
                         code, cap)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(replays):
            graph.replay()
        b.record()
        torch.cuda.synchronize(dev)
        dev_us = a.elapsed_time(b) * 1e3 / (replays * graph_launches)
        # host time of one call (launches queue up; the GPU keeps pace or falls behind)
        t0 = time.perf_counter()
        for _ in range(200):
            launch()
        host_us = (time.perf_counter() - t0) * 1e6 / 200
        torch.cuda.synchronize(dev)
        out[name] = {"workload": f"{name}: B={w.B} H={w.H} S={w.S_q} d={w.d} {w.dtype} "
                                 f"{'causal' if causal else 'full'}",
                     "us": pc["median_ms"] * 1e3, "p10_us": pc["p10_ms"] * 1e3,
                     "p90_us": pc["p90_ms"] * 1e3, "bytes": w.io_bytes(),
                     "gbs": w.io_bytes() / t / 1e9, "tflops": w.flops(causal) / t / 1e12,
                     "l2": "256 MB flush before each launch" if name == "c1" else "no flush",
                     "device_us": dev_us, "device_gbs": w.io_bytes() / (dev_us * 1e-6) / 1e9,
                     "device_tflops": w.flops(causal) / (dev_us * 1e-6) / 1e12,
                     "device_how": f"{graph_launches} launches back to back in one CUDA graph, "
                                   f"{replays} replays, L2 not flushed",
                     "host_us_per_call": host_us}
    out["c1"]["note"] = "latency-bound (66 KB, one tile): the roofline fraction is not meaningful"
    return out


def measure_bwd(dev, stream, w, q, k, v, iters: int = 10):
    """Backward (dQ, dK, dV) on the benchmark workload, both masking modes.

    FLOPs per call are counted as 2.5 forwards (the five S_q×S_k×d products
    dV = Pᵀ·dO, dP = dO·Vᵀ, dQ = dS·K, dK = dSᵀ·Q and the recomputed Q·Kᵀ),
    halved when causal; the kernels execute seven such products (dQ has its
    own pass that recomputes Q·Kᵀ and dO·Vᵀ, so no atomics are needed).
    """
    import torch

    from exact_attention_53_gb300 import attn_bwd, attn_bwd_workspace_size, attn_fwd
    from exact_attention_53_gb300.binding import ATTN_DTYPE_BF16
    from exact_attention_53_gb300.workloads import make_qkv

    B, H, S_q, S_k, d = w.B, w.H, w.S_q, w.S_k, w.d
    dout = make_qkv(B, H, S_q, 1, d, w.dtype, seed=w.seed + 100)[0].to(dev)
    ws = attn_bwd_workspace_size(B, H, S_q, S_k, d, ATTN_DTYPE_BF16)
    work = torch.empty(ws, dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    res = {}
    for causal in (False, True):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=dev)
        attn_fwd(q, k, v, o, lse, B, H, S_q, S_k, d, int(causal), w.scale, ATTN_DTYPE_BF16, stream)

        def call():
            attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, S_q, S_k, d, int(causal), w.scale,
                     ATTN_DTYPE_BF16, work, ws, stream)

        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)]
        for a, b in ev:
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        flops = 2.5 * w.flops(causal)
        res["causal" if causal else "full"] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}
    res["flops_convention"] = "2.5 x forward (five S_q x S_k x d products), halved when causal"
    res["gpu_launches_per_call"] = 3
    res["calls_timed"] = iters
    return res


def run_gpu(args, rank, world):
    import torch

    from exact_attention_53_gb300 import attn_fwd, attn_fwd_host, attn_get_device_status
    from exact_attention_53_gb300.binding import ATTN_DTYPE_BF16, load_library
    from exact_attention_53_gb300.build import build
    from exact_attention_53_gb300.workloads import WORKLOADS, workload_qkv

    local = _env_int("LOCAL_RANK", 0)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        build()
    if world > 1:
        torch.distributed.barrier()
    load_library()

    w = WORKLOADS[WORKLOAD]
    B, H, S_q, S_k, d = w.B, w.H, w.S_q, w.S_k, w.d
    q_h, k_h, v_h = workload_qkv(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S_q), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = {False: w.flops(False), True: w.flops(True)}
    flops_step = flops[False] + flops[True]

    def launch(causal):
        attn_fwd(q, k, v, o, lse, B, H, S_q, S_k, d, int(causal), w.scale, ATTN_DTYPE_BF16, stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    sampler.start()
    # Untimed warm-up: at least W steps, and at least ~0.4 s so the clocks have
    # ramped and the sampler has seen the GPU under this load.
    t_w = time.time()
    warm = 0
    while warm < args.warmup or time.time() - t_w < 0.4:
        launch(False)
        launch(True)
        warm += 1
        if warm % 8 == 0:
            torch.cuda.synchronize(dev)
    attn_get_device_status(stream)
    barrier()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        launch(False)
        ev[i][1].record(stream)
        launch(True)
        ev[i][2].record(stream)
    end.record(stream)
    barrier()
    t_wall1 = time.time()
    total_ms = start.elapsed_time(end)
    full_ms = [e[0].elapsed_time(e[1]) for e in ev]
    causal_ms = [e[1].elapsed_time(e[2]) for e in ev]
    attn_get_device_status(stream)

    total_ms = max_over_ranks(total_ms, world, dev)
    value = replica_throughput(flops_step, args.steps, world, total_ms)

    # ---- e2e: host buffers in, host buffers out, through attn_fwd_host
    qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    op = torch.empty_like(qp).pin_memory()
    lp = torch.empty((B, H, S_q), dtype=torch.float32).pin_memory()
    q2, k2, v2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def e2e_launch(causal):
        attn_fwd_host(qp, kp, vp, op, lp, q2, k2, v2, o, lse, B, H, S_q, S_k, d, int(causal),
                      w.scale, ATTN_DTYPE_BF16, stream)

    for _ in range(args.warmup):
        e2e_launch(False)
        e2e_launch(True)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_launch(False)
        e2e_launch(True)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = replica_throughput(flops_step, args.steps, world, e2e_ms)
    in_bytes = q.numel() * 2 + k.numel() * 2 + v.numel() * 2
    out_bytes = o.numel() * 2 + lse.numel() * 4
    splitkv = measure_splitkv(dev, stream)
    backward = measure_bwd(dev, stream, w, q, k, v)
    short = measure_short(dev, stream)
    long_ = measure_long(dev, stream)
    from exact_attention_53_gb300.binding import probe_ex2_rate
    ex2_peak = probe_ex2_rate()
    attn_get_device_status(stream)
    sampler.stop()

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    full_avg = statistics.mean(full_ms)
    causal_avg = statistics.mean(causal_ms)
    achieved = flops[False] / (full_avg * 1e-3) / 1e12
    achieved_c = flops[True] / (causal_avg * 1e-3) / 1e12
    clocks = sampler.summary(t_wall0, t_wall1)
    traffic = measured_traffic("attn_fwd_d128_bf16_full_c3")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "warmup_steps_run": warm,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: B={B} H={H} S_q=S_k={S_q} d={d} bf16, one full + one "
                               f"causal forward per step, scale=1/sqrt(128), Q,K~N(0,1) V~U(-1,1)",
                   "global_batch": B * world, "seq_len": S_q,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (Q+K+V = 201 MB > 129 MB), no flush"},
        "modes": {"full": {"ms": full_avg, "tflops": achieved, "frac_of_peak": achieved / peak,
                           **percentiles(full_ms)},
                  "causal": {"ms": causal_avg, "tflops": achieved_c,
                             "frac_of_peak": achieved_c / peak, **percentiles(causal_ms)}},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "attn_fwd_kernel<128,bf16,full>",
                     "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
                     if peak_src == "measured" else "fallback 1.9 PFLOP/s"},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 2 * in_bytes,
                "d2h_bytes_per_step": 2 * out_bytes},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    splitkv["roofline"] = {"bound": "hbm", "achieved": splitkv["gbs"], "peak": hbm, "unit": "GB/s",
                           "frac": splitkv["gbs"] / hbm,
                           "traffic": measured_traffic("attn_fwd_splitkv_d128_bf16_decode"),
                           "kernel": "attn_fwd_kernel<128,bf16,full,split> + attn_combine_kernel",
                           "peak_source": f"{peak_src} copy bandwidth (hbm_gbs)"}
    line["splitkv"] = splitkv
    for mode in ("full", "causal"):
        backward[mode]["frac_of_peak"] = backward[mode]["tflops"] / peak
    backward["roofline"] = {"bound": "tensor", "achieved": backward["full"]["tflops"], "peak": peak,
                            "unit": "TFLOP/s", "frac": backward["full"]["tflops"] / peak,
                            "traffic": measured_traffic("attn_bwd_d128_bf16_full_c3"),
                            "kernel": "attn_bwd_prep + attn_bwd_dkdv + attn_bwd_dq <128,bf16,full>",
                            "peak_source": "measured bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
                            if peak_src == "measured" else "fallback 1.9 PFLOP/s"}
    backward["workload"] = f"{WORKLOAD}: B={B} H={H} S_q=S_k={S_q} d={d} bf16, dO~N(0,1)"
    line["backward"] = backward
    line["short"] = short
    line["long"] = long_
    # Secondary ceiling: exponentials (S_q·S_k per head, halved causal) per second against the
    # ex2.approx throughput of the MUFU pipe measured by attn_probe_ex2 in this run.
    exps = {False: B * H * S_q * S_k, True: B * H * S_q * S_k / 2}
    line["exp_rate"] = {
        "probe_ex2_per_s": ex2_peak,
        "full": {"ex2_per_s": exps[False] / (full_avg * 1e-3),
                 "frac": exps[False] / (full_avg * 1e-3) / ex2_peak},
        "causal": {"ex2_per_s": exps[True] / (causal_avg * 1e-3),
                   "frac": exps[True] / (causal_avg * 1e-3) / ex2_peak}}
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline()
        line["cpu_baseline"]["per_config"] = cpu_per_config()
    print(json.dumps(line), flush=True)

# ------------------------------------------------------------------ sweeps
# Range-count and grouped-head sweeps of the split-KV forward (``--sweep``):
# µs per call, printed as markdown tables, outside the benchmark's timed steps.
SWEEP_SHAPES = [(2, 16, 1, 32768, 128), (1, 8, 1, 131072, 128), (8, 32, 1, 8192, 128),
                (2, 16, 1, 32768, 64), (2, 8, 1, 32768, 256), (2, 16, 128, 32768, 128)]
SWEEP_SPLITS = (0, 2, 4, 8, 16, 32)
GQA_SHAPES = [(8, 32, 8, 1, 8192, 128), (2, 64, 8, 1, 32768, 128), (4, 32, 4, 4, 16384, 128),
              (16, 32, 8, 1, 4096, 128), (2, 32, 8, 1, 65536, 64)]


def _mean_ms(fn, iters=20):
    import torch

    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def split_sweep():
    """µs per call of the one-pass and split-KV forwards (bf16, full attention)."""
    import torch

    from exact_attention_53_gb300 import (attn_fwd_splitkv_plan, attn_get_device_status, fwd,
                                          fwd_splitkv)
    from exact_attention_53_gb300.workloads import make_qkv

    dev = torch.device("cuda")
    print("| shape (B, H, S_q, S_k, d) | one-pass | " +
          " | ".join("auto (ranges)" if n == 0 else str(n) for n in SWEEP_SPLITS) + " |")
    for B, H, S_q, S_k, d in SWEEP_SHAPES:
        q, k, v = (t.to(dev) for t in make_qkv(B, H, S_q, S_k, d, "bf16", seed=1))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=dev)
        cells = [f"{1e3 * _mean_ms(lambda: fwd(q, k, v, out=o, lse=lse)):.1f}"]
        for n in SWEEP_SPLITS:
            used, ws = attn_fwd_splitkv_plan(B, H, S_q, S_k, d, 1, n)
            work = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
            t = 1e3 * _mean_ms(lambda: fwd_splitkv(q, k, v, n_split=n, workspace=work, out=o,
                                                   lse=lse))
            cells.append(f"{t:.1f} ({used})" if n == 0 else f"{t:.1f}")
        attn_get_device_status()
        print(f"| {B}, {H}, {S_q}, {S_k}, {d} | " + " | ".join(cells) + " |", flush=True)


def gqa_sweep():
    """Decoding with grouped key/value heads: one-pass vs split-KV with packed heads."""
    import torch

    from exact_attention_53_gb300 import attn_get_device_status, fwd_general, fwd_splitkv_general
    from exact_attention_53_gb300.workloads import make_qkv

    dev = torch.device("cuda")
    print("| shape (B, H, H_kv, S_q, S_k, d) | one-pass µs | split-KV µs (auto) | split GB/s |")
    print("|---|---|---|---|")
    for B, H, H_kv, S_q, S_k, d in GQA_SHAPES:
        q = make_qkv(B, H, S_q, 1, d, "bf16", seed=2)[0].to(dev)
        _, k, v = (t.to(dev) for t in make_qkv(B, H_kv, 1, S_k, d, "bf16", seed=3))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=dev)
        work = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
        t1 = 1e3 * _mean_ms(lambda: fwd_general(q, k, v, out=o, lse=lse))
        t2 = 1e3 * _mean_ms(lambda: fwd_splitkv_general(q, k, v, n_split=0, workspace=work,
                                                         out=o, lse=lse))
        by = 2 * (2 * B * H * S_q * d + 2 * B * H_kv * S_k * d) + 4 * B * H * S_q
        attn_get_device_status()
        print(f"| {B}, {H}, {H_kv}, {S_q}, {S_k}, {d} | {t1:.1f} | {t2:.1f} | {by / t2 / 1e3:.0f} |",
              flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the ~12 s oracle timing on the host cores")
    ap.add_argument("--sweep", choices=["split", "gqa"], default=None,
                    help="print a split-KV range-count or grouped-head table instead")
    args = ap.parse_args()
    if args.sweep:
        (split_sweep if args.sweep == "split" else gqa_sweep)()
        return
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(_env_int("LOCAL_RANK", 0))
        torch.distributed.init_process_group("nccl")
    try:
        run_gpu(args, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
