"""Run the attention forward on a named workload (for profiling).

    python -m exact_attention_53_gb300.run --workload c3 --causal 0 --iters 2
    python -m exact_attention_53_gb300.run --workload decode --split 0 --iters 2
    python -m exact_attention_53_gb300.run --split-sweep
    python -m exact_attention_53_gb300.run --gqa-sweep
    python -m exact_attention_53_gb300.run --workload c3 --causal 1 --bwd --iters 3

Inputs are the seeded synthetic ones of ``workloads``; the forward is
launched ``--iters`` times on the current stream, then the device status is
checked.  Prints the device time per launch and the TFLOP/s (the best
launch), or with ``--split N`` (split-KV, N ranges, 0 = automatic) the HBM
GB/s of the algorithmic bytes.  ``--split-sweep`` times the split-KV forward
over a grid of short-query shapes and range counts beside the one-pass kernel.
``--bwd`` runs the forward once, then times the backward (dQ, dK, dV for a
seeded dO) and prints TFLOP/s counted as 2.5 forwards (five S_q×S_k×d
products).
"""

from __future__ import annotations

import argparse

import torch

from . import (attn_fwd_splitkv_plan, attn_get_device_status, bwd, fwd, fwd_general, fwd_splitkv,
               fwd_splitkv_general)
from .workloads import WORKLOADS, make_qkv, workload_qkv


SWEEP_SHAPES = [(2, 16, 1, 32768, 128), (1, 8, 1, 131072, 128), (8, 32, 1, 8192, 128),
                (2, 16, 1, 32768, 64), (2, 8, 1, 32768, 256), (2, 16, 128, 32768, 128)]
SWEEP_SPLITS = (0, 2, 4, 8, 16, 32)


def _mean_ms(fn, iters=20):
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
            t = 1e3 * _mean_ms(lambda: fwd_splitkv(q, k, v, n_split=n, workspace=work, out=o, lse=lse))
            cells.append(f"{t:.1f} ({used})" if n == 0 else f"{t:.1f}")
        attn_get_device_status()
        print(f"| {B}, {H}, {S_q}, {S_k}, {d} | " + " | ".join(cells) + " |", flush=True)


GQA_SHAPES = [(8, 32, 8, 1, 8192, 128), (2, 64, 8, 1, 32768, 128), (4, 32, 4, 4, 16384, 128),
              (16, 32, 8, 1, 4096, 128), (2, 32, 8, 1, 65536, 64)]


def gqa_sweep():
    """Decoding with grouped key/value heads: one-pass vs split-KV with packed heads."""
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


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="c3", choices=sorted(WORKLOADS))
    ap.add_argument("--causal", type=int, default=None, help="0/1; default: the workload's first mode")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--heads", type=int, default=None, help="override B·H (keeps B=1) for a smaller case")
    ap.add_argument("--split", type=int, default=None,
                    help="run the split-KV forward with this many ranges (0 = automatic)")
    ap.add_argument("--split-sweep", action="store_true",
                    help="time split-KV over short-query shapes and range counts")
    ap.add_argument("--bwd", action="store_true", help="time the backward instead of the forward")
    ap.add_argument("--gqa-sweep", action="store_true",
                    help="time decoding with grouped key/value heads, one-pass vs split-KV")
    args = ap.parse_args(argv)
    if args.split_sweep:
        split_sweep()
        return 0
    if args.gqa_sweep:
        gqa_sweep()
        return 0
    w = WORKLOADS[args.workload]
    causal = bool(w.causal[0] if args.causal is None else args.causal)
    if args.heads:
        q, k, v = make_qkv(1, args.heads, w.S_q, w.S_k, w.d, w.dtype, w.seed, w.qk_dist, w.v_dist)
        bh = args.heads
    else:
        q, k, v = workload_qkv(w)
        bh = w.B * w.H
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.iters + 1)]
    if args.bwd:
        dout = make_qkv(q.shape[0], q.shape[1], w.S_q, 1, w.d, w.dtype, w.seed + 100)[0].to(dev)
        fwd(q, k, v, causal=causal, scale=w.scale, out=o, lse=lse)
        ev[0].record()
        for i in range(args.iters):
            bwd(q, k, v, o, lse, dout, causal=causal, scale=w.scale)
            ev[i + 1].record()
        attn_get_device_status()
        ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.iters)]
        flops = 10.0 * bh * w.S_q * w.S_k * w.d / (2 if causal else 1)
        print(f"{args.workload} bwd causal={int(causal)} B*H={bh}: per-call ms {['%.3f' % x for x in ms]}"
              f" best {flops / min(ms) / 1e9:.1f} TFLOP/s")
        return 0
    if args.split is not None:
        n, ws = attn_fwd_splitkv_plan(1 if args.heads else w.B, bh if args.heads else w.H, w.S_q,
                                      w.S_k, w.d, 1 if w.dtype == "bf16" else 0, args.split)
        work = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
    ev[0].record()
    for i in range(args.iters):
        if args.split is not None:
            fwd_splitkv(q, k, v, n_split=args.split, scale=w.scale, workspace=work, out=o, lse=lse)
        else:
            fwd(q, k, v, causal=causal, scale=w.scale, out=o, lse=lse)
        ev[i + 1].record()
    attn_get_device_status()
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.iters)]
    if args.split is not None:
        by = 2 * bh * (2 * w.S_q + 2 * w.S_k) * w.d + 4 * bh * w.S_q
        print(f"{args.workload} split-KV n_split={n} B*H={bh}: per-call ms {['%.4f' % x for x in ms]}"
              f" best {by / min(ms) / 1e6:.0f} GB/s")
        return 0
    flops = 4.0 * bh * w.S_q * w.S_k * w.d / (2 if causal else 1)
    best = min(ms)
    print(f"{args.workload} causal={int(causal)} B*H={bh}: per-launch ms {['%.3f' % x for x in ms]}"
          f" best {flops / best / 1e9:.1f} TFLOP/s")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
