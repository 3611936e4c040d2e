"""Run the attention forward on a named workload (for profiling).

    python -m exact_attention_53_gb300.run --workload c3 --causal 0 --iters 2
    python -m exact_attention_53_gb300.run --workload decode --split 0 --iters 2
    python -m exact_attention_53_gb300.run --workload c3 --causal 1 --bwd --iters 3

Inputs are the seeded synthetic ones of ``workloads``; the forward is
launched ``--iters`` times on the current stream, then the device status is
checked.  Prints the device time per launch and the TFLOP/s (the best
launch), or with ``--split N`` (split-KV, N ranges, 0 = automatic) the HBM
GB/s of the algorithmic bytes.  ``--bwd`` runs the forward once, then times the backward (dQ, dK, dV for a
seeded dO) and prints TFLOP/s counted as 2.5 forwards (five S_q×S_k×d
products).
"""

from __future__ import annotations

import argparse

import torch

from . import attn_fwd_splitkv_plan, attn_get_device_status, bwd, fwd, fwd_splitkv
from .workloads import WORKLOADS, make_qkv, workload_qkv


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="c3", choices=sorted(WORKLOADS))
    ap.add_argument("--causal", type=int, default=None, help="0/1; default: the workload's first mode")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--heads", type=int, default=None, help="override B·H (keeps B=1) for a smaller case")
    ap.add_argument("--split", type=int, default=None,
                    help="run the split-KV forward with this many ranges (0 = automatic)")
    ap.add_argument("--bwd", action="store_true", help="time the backward instead of the forward")
    args = ap.parse_args(argv)
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
