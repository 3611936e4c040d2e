"""GPU parity of the split-KV forward (through the C ABI) against the fp64 oracle.

The split path cuts the keys into ranges, writes per-range partial O/LSE to a
workspace and merges them with a second kernel; its result must match the
oracle within the same tolerances as the one-pass forward, for every head
dimension and dtype, for range counts that divide the key tiles evenly or not,
for more ranges than a warp has lanes, and with a workspace that starts out
holding garbage.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_53_gb300 import (attn_fwd_splitkv, attn_fwd_splitkv_plan,
                                      attn_get_device_status, fwd, fwd_splitkv)
from exact_attention_53_gb300.binding import ATTN_DTYPE_BF16
from exact_attention_53_gb300.workloads import WORKLOADS, make_qkv, workload_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
DTYPE_CODE = {"f16": 0, "bf16": 1}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_53_gb300.build import build
    build()
    yield
    attn_get_device_status()


# (B, H, S_q, S_k): one decode row, a ragged query tile, a full 128-row tile,
# two query blocks (S_q > 256), a key length just past a tile boundary.
SHAPES = [(1, 3, 1, 5000), (2, 2, 37, 9000), (1, 2, 128, 4096), (1, 1, 300, 2000),
          (1, 2, 5, 1153)]


@pytest.mark.parametrize("n_split", [1, 3, 7, 0], ids=lambda n: f"split{n}")
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_splitkv_matches_oracle(d, dtype, shape, n_split):
    B, H, S_q, S_k = shape
    q, k, v = make_qkv(B, H, S_q, S_k, d, dtype, seed=S_q * 131 + S_k * 7 + d + n_split)
    scale = 1 / math.sqrt(d)
    o, lse = fwd_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), n_split=n_split, scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=scale)
    assert_parity(o, lse, ro, rl, dtype, f"split-KV d={d} {dtype} {shape} n_split={n_split}")


def test_more_ranges_than_lanes():
    """128 key tiles in 64 ranges of 2: the merge's max runs over more than 32 ranges."""
    B, H, S_q, S_k, d = 1, 2, 3, 16384, 128
    q, k, v = make_qkv(B, H, S_q, S_k, d, "bf16", seed=21)
    n, _ = attn_fwd_splitkv_plan(B, H, S_q, S_k, d, ATTN_DTYPE_BF16, 100)
    assert n == 64
    o, lse = fwd_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), n_split=100)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=1 / math.sqrt(d))
    assert_parity(o, lse, ro, rl, "bf16", "64 ranges")


def test_ranges_with_very_different_maxima():
    """Logits ramp along the keys, so the ranges' LSEs differ by tens of nats."""
    B, H, S_q, S_k, d = 1, 2, 20, 6000, 128
    q, k, v = make_qkv(B, H, S_q, S_k, d, "bf16", seed=22)
    ramp = torch.linspace(-4, 4, S_k).view(1, 1, S_k, 1)
    k = (k.float() * 0.2 + ramp * q.float().mean(dim=2, keepdim=True)).to(torch.bfloat16)
    for n_split in (2, 5, 47):
        o, lse = fwd_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), n_split=n_split, scale=1.0)
        torch.cuda.synchronize()
        ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=1.0)
        assert_parity(o, lse, ro, rl, "bf16", f"ramped logits n_split={n_split}")


def test_workspace_needs_no_clearing_and_stays_in_bounds():
    """A NaN-filled workspace gives the same result; nothing past its size is written."""
    B, H, S_q, S_k, d = 2, 3, 9, 3000, 64
    q, k, v = make_qkv(B, H, S_q, S_k, d, "f16", seed=23)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    n, ws = attn_fwd_splitkv_plan(B, H, S_q, S_k, d, DTYPE_CODE["f16"], 6)
    assert n == 6 and ws > 0
    pad = 4096
    buf = torch.full((ws + 2 * pad,), 0xFF, dtype=torch.uint8, device=DEV)   # NaN bytes
    work = buf[pad:pad + ws]
    o_buf = torch.full((B * H * S_q * d + 2 * pad,), 7.0, dtype=torch.float16, device=DEV)
    o = o_buf[pad:pad + B * H * S_q * d]
    lse = torch.empty((B, H, S_q), dtype=torch.float32, device=DEV)
    attn_fwd_splitkv(qd, kd, vd, o, lse, B, H, S_q, S_k, d, 1 / math.sqrt(d), DTYPE_CODE["f16"],
                     6, work, ws)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 0xFF) and torch.all(buf[pad + ws:] == 0xFF)
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[pad + o.numel():] == 7.0)
    ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=1 / math.sqrt(d))
    assert_parity(o.view(B, H, S_q, d), lse, ro, rl, "f16", "NaN workspace")


def test_agrees_with_one_pass_forward():
    """Split and one-pass results agree with each other within the dtype's tolerance."""
    q, k, v = make_qkv(2, 4, 64, 8192, 128, "bf16", seed=24)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = fwd(qd, kd, vd)
    o2, l2 = fwd_splitkv(qd, kd, vd, n_split=8)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_repeated_calls_are_deterministic():
    q, k, v = make_qkv(1, 4, 16, 7000, 128, "bf16", seed=25)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = fwd_splitkv(qd, kd, vd, n_split=5)
    o2, l2 = fwd_splitkv(qd, kd, vd, n_split=5)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_workload_full_size():
    """The decode workload at full size with the automatic range count, every row."""
    w = WORKLOADS["decode"]
    q, k, v = workload_qkv(w)
    n, _ = attn_fwd_splitkv_plan(w.B, w.H, w.S_q, w.S_k, w.d, ATTN_DTYPE_BF16, 0)
    assert n > 1
    o, lse = fwd_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), n_split=0, scale=w.scale)
    torch.cuda.synchronize()
    assert np.isfinite(o.float().cpu().numpy()).all()
    ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=w.scale)
    assert_parity(o, lse, ro, rl, w.dtype, "decode workload")


# ------------------------------------------------- grouped heads, general layouts
from exact_attention_53_gb300 import fwd_splitkv_general  # noqa: E402


def _gqa_inputs(B, H, H_kv, S_q, S_k, d, dtype, seed):
    q = make_qkv(B, H, S_q, 1, d, dtype, seed=seed)[0]
    _, k, v = make_qkv(B, H_kv, 1, S_k, d, dtype, seed=seed + 1)
    return q, k, v


def _bshd(t):
    return t.transpose(1, 2).contiguous().transpose(1, 2)


# (B, H, H_kv, S_q, S_k): decode with groups of 4 and 8 (packed), 16·8 = 128
# rows exactly, MQA, and 40·4 = 160 rows (too many to pack: one head per tile)
GQA_SHAPES = [(2, 32, 8, 1, 5000), (1, 16, 2, 1, 9000), (1, 16, 2, 16, 3000), (2, 16, 1, 1, 4100),
              (1, 8, 2, 40, 2000), (16, 32, 8, 1, 4096)]


@pytest.mark.parametrize("n_split", [1, 3, 0], ids=lambda n: f"split{n}")
@pytest.mark.parametrize("shape", GQA_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_splitkv_grouped_heads_match_oracle(d, dtype, shape, n_split):
    B, H, H_kv, S_q, S_k = shape
    q, k, v = _gqa_inputs(B, H, H_kv, S_q, S_k, d, dtype, seed=S_k + H * 3 + d)
    scale = 1 / math.sqrt(d)
    o = _bshd(torch.empty((B, H, S_q, d), dtype=q.dtype, device=DEV))
    o, lse = fwd_splitkv_general(_bshd(q.to(DEV)), _bshd(k.to(DEV)), _bshd(v.to(DEV)),
                                 n_split=n_split, scale=scale, out=o)
    torch.cuda.synchronize()
    g = H // H_kv
    ro, rl = oracle.attention_forward(q, k.repeat_interleave(g, dim=1),
                                      v.repeat_interleave(g, dim=1), causal=False, scale=scale)
    assert_parity(o, lse, ro, rl, dtype, f"grouped split-KV d={d} {dtype} {shape} n={n_split}")


def test_packed_groups_match_repeated_heads_bitwise():
    """Packing a group's heads into one tile changes no row's arithmetic."""
    B, H, H_kv, S_q, S_k, d = 2, 32, 8, 1, 8192, 128
    q, k, v = _gqa_inputs(B, H, H_kv, S_q, S_k, d, "bf16", seed=71)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = fwd_splitkv_general(qd, kd, vd, n_split=5)
    o2, l2 = fwd_splitkv(qd, kd.repeat_interleave(4, dim=1).contiguous(),
                         vd.repeat_interleave(4, dim=1).contiguous(), n_split=5)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
