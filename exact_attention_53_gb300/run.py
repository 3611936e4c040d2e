"""Run the attention forward on a named workload (for profiling).

    python -m exact_attention_53_gb300.run --workload c3 --causal 0 --iters 2

Inputs are the seeded synthetic ones of ``workloads``; the forward is
launched ``--iters`` times on the current stream, then the device status is
checked.  Prints the mean device time per launch and the TFLOP/s.
"""

from __future__ import annotations

import argparse

import torch

from . import attn_get_device_status, fwd
from .workloads import WORKLOADS, make_qkv, workload_qkv


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="c3", choices=sorted(WORKLOADS))
    ap.add_argument("--causal", type=int, default=None, help="0/1; default: the workload's first mode")
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--heads", type=int, default=None, help="override B·H (keeps B=1) for a smaller case")
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
    ev[0].record()
    for i in range(args.iters):
        fwd(q, k, v, causal=causal, scale=w.scale, out=o, lse=lse)
        ev[i + 1].record()
    attn_get_device_status()
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.iters)]
    flops = 4.0 * bh * w.S_q * w.S_k * w.d / (2 if causal else 1)
    best = min(ms)
    print(f"{args.workload} causal={int(causal)} B*H={bh}: per-launch ms {['%.3f' % x for x in ms]}"
          f" best {flops / best / 1e9:.1f} TFLOP/s")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
