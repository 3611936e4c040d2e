"""Seeded synthetic inputs for the attention forward.

This module only draws random numbers: it holds none of the attention
arithmetic, and both the CUDA path's tests/bench and the CPU oracle take their
inputs from it.  Inputs are drawn on the CPU in float32 from
``torch.Generator().manual_seed(seed)`` (Q first, then K, then V), cast to the
workload dtype, and only then copied to a device, so every consumer sees the
same rounded values.

The five workloads c1..c5 follow the configurations the attention page's
FlashAttention-3 plan is sized for (oxicuda-dnn 0.1.8 hopper.rs,
``SUPPORTED_HEAD_DIMS`` = 64/128/256 and ``default_for`` tile sizes), with the
shapes, value distributions and seeds fixed here; ``decode`` is the short-query,
long-key shape the split-KV forward is for.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S_q: int
    S_k: int
    d: int
    dtype: str              # "f16" | "bf16"
    causal: tuple           # the masking modes this workload is run in
    scale: float
    qk_dist: str            # "normal" | "normal2" (2·N(0,1))
    v_dist: str             # "normal" | "uniform" (U(-1,1))
    seed: int

    def flops(self, causal: bool) -> float:
        """4·B·H·S_q·S_k·d, halved when causal (the metric's convention)."""
        f = 4.0 * self.B * self.H * self.S_q * self.S_k * self.d
        return f / 2 if causal else f

    def io_bytes(self) -> int:
        """Q, K, V read once, O written once, plus the fp32 LSE."""
        e = 2
        return (e * self.B * self.H * (2 * self.S_q + 2 * self.S_k) * self.d
                + 4 * self.B * self.H * self.S_q)


WORKLOADS = {
    "c1": Workload("c1", 1, 1, 128, 128, 64, "f16", (False,), 1 / math.sqrt(64),
                   "normal", "normal", 1001),
    "c2": Workload("c2", 4, 16, 1024, 1024, 64, "bf16", (True,), 1 / 8,
                   "normal", "normal", 1002),
    "c3": Workload("c3", 2, 32, 4096, 4096, 128, "bf16", (False, True), 1 / math.sqrt(128),
                   "normal", "uniform", 1003),
    "c4": Workload("c4", 1, 16, 16384, 16384, 128, "bf16", (True,), 1 / math.sqrt(128),
                   "normal2", "normal", 1004),
    "c5": Workload("c5", 2, 8, 8192, 8192, 256, "bf16", (False,), 1 / 16,
                   "normal", "normal", 1005),
    # Decoding step against a long key cache: one query row per head and few
    # heads, so B·H alone gives far fewer work units than SMs (split-KV).
    "decode": Workload("decode", 2, 16, 1, 32768, 128, "bf16", (False,), 1 / math.sqrt(128),
                       "normal", "normal", 1006),
}

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


def _draw(g: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "normal2":
        return 2.0 * torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    raise ValueError(f"unknown distribution {dist!r}")


def make_qkv(B: int, H: int, S_q: int, S_k: int, d: int, dtype: str = "bf16",
             seed: int = 0, qk_dist: str = "normal", v_dist: str = "normal"):
    """Q [B,H,S_q,d], K and V [B,H,S_k,d] on the CPU, in ``dtype``."""
    g = torch.Generator().manual_seed(seed)
    td = TORCH_DTYPE[dtype]
    q = _draw(g, (B, H, S_q, d), qk_dist).to(td)
    k = _draw(g, (B, H, S_k, d), qk_dist).to(td)
    v = _draw(g, (B, H, S_k, d), v_dist).to(td)
    return q, k, v


def workload_qkv(w: Workload):
    """The seeded inputs of a named workload."""
    return make_qkv(w.B, w.H, w.S_q, w.S_k, w.d, w.dtype, w.seed, w.qk_dist, w.v_dist)
