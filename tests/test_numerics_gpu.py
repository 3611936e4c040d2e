"""GPU parity at the edges of the arithmetic: growing logits, fp16 range, negative scale.

Every case goes through the C ABI and is compared element by element with the
fp64 oracle at the stated tolerances (bf16 |ΔO| <= 1e-2 + 1e-2·|O|, f16
|ΔO| <= 4e-3, |ΔLSE| <= 1e-3).

* Growing logits.  The kernel exponentiates later key tiles against a running
  maximum that may be stale and only redoes a row when the tile's sum of
  exponentials passes a bound.  In fp16 each p must stay below 65504 (the
  packed P would round to +inf), so a later key whose logit exceeds the first
  tile's maximum by 12 or 13 nats (e^12 ≈ 1.6e5, e^13 ≈ 4.4e5: above 65504,
  below the bf16 bound 2^20) must trigger the redo.  All keys but one are nearly
  orthogonal to every query (logits within a few tenths of 0); one key, in the
  second tile (or, as a control, in the first), has q·k = 12 or 13 at scale 1.
* fp16 near its largest value.  Q, K and V of magnitude 5e4–6.5e4 (logits kept
  O(1) by the scale).  O is linear in V, so the fp16 tolerance scales with V:
  O / max|V| is compared at 4e-3.
* Negative scale.  scale = −0.1 in both masks, the split-KV path and the
  bottom-right mask.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_53_gb300 import attn_get_device_status, fwd, fwd_general, fwd_splitkv
from exact_attention_53_gb300.binding import ATTN_MASK_CAUSAL_BOTTOM_RIGHT
from exact_attention_53_gb300.workloads import TORCH_DTYPE, make_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_53_gb300.build import build
    build()
    yield
    attn_get_device_status()


def _growth_inputs(B, H, S_q, S_k, d, dtype, excess, specials, seed):
    """Q rows (1, 0.1·N(0,1)...), K rows (0, 0.1·N(0,1)...) except the keys in `specials`,
    whose first coordinate is `excess`: at scale 1 those keys' logits are excess + O(0.2),
    every other logit O(0.2)."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, S_q, d, generator=g) * 0.1
    q[..., 0] = 1.0
    k = torch.randn(B, H, S_k, d, generator=g) * 0.1
    k[..., 0] = 0.0
    for j in specials:
        k[..., j, 0] = float(excess)
    v = torch.randn(B, H, S_k, d, generator=g)
    td = TORCH_DTYPE[dtype]
    return q.to(td), k.to(td), v.to(td)


@pytest.mark.parametrize("special", [200, 100], ids=["second_tile", "first_tile"])
@pytest.mark.parametrize("excess", [12, 13])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_logit_growth_past_the_fp16_range(d, dtype, causal, excess, special):
    # key 200 sits in the second key tile: every query tile meets it after key tile 0;
    # key 100 sits in the first tile (rows that see it take its maximum first)
    q, k, v = _growth_inputs(1, 2, 512, 512, d, dtype, excess, [special],
                             seed=500 + d + excess + special)
    o, lse = fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=1.0)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=causal, scale=1.0)
    assert_parity(o, lse, ro, rl, dtype,
                  f"growth {excess} at key {special} d={d} {dtype} causal={causal}")


@pytest.mark.parametrize("excess", [12, 13])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_logit_growth_in_split_ranges(d, dtype, excess):
    # 8 key tiles in 2 ranges; each range meets one large key in its second tile
    q, k, v = _growth_inputs(1, 2, 64, 1024, d, dtype, excess, [200, 700], seed=520 + d + excess)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = fwd_splitkv(qd, kd, vd, n_split=2, scale=1.0)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=1.0)
    assert_parity(o, lse, ro, rl, dtype, f"split growth {excess} d={d} {dtype}")


def _signed_uniform(g, shape, lo, hi):
    mag = lo + (hi - lo) * torch.rand(shape, generator=g, dtype=torch.float64)
    sign = torch.where(torch.rand(shape, generator=g) < 0.5, -1.0, 1.0).double()
    return mag * sign


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_f16_inputs_near_the_largest_value(d, causal):
    B, H, S = 1, 2, 384
    g = torch.Generator().manual_seed(540 + d)
    q = _signed_uniform(g, (B, H, S, d), 5.0e4, 6.0e4).to(torch.float16)
    k = _signed_uniform(g, (B, H, S, d), 5.0e4, 6.0e4).to(torch.float16)
    v = _signed_uniform(g, (B, H, S, d), 5.5e4, 65504.0).to(torch.float16)
    assert torch.isfinite(v.float()).all() and v.float().abs().max() <= 65504
    scale = 1.0 / (5.5e4 ** 2 * math.sqrt(d))      # logits of order one
    o, lse = fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=causal, scale=scale)
    vmax = float(v.float().abs().max())
    o64 = o.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(o64).all()
    assert_parity(o64 / vmax, lse, ro / vmax, rl, "f16", f"near 65504 d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_negative_scale(d, dtype, causal):
    q, k, v = make_qkv(1, 2, 300, 300, d, dtype, seed=560 + d)
    o, lse = fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=-0.1)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=causal, scale=-0.1)
    assert_parity(o, lse, ro, rl, dtype, f"scale=-0.1 d={d} {dtype} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_negative_scale_split_and_bottom_right(d):
    q, k, v = make_qkv(1, 4, 5, 3000, d, "bf16", seed=580 + d)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = fwd_splitkv(qd, kd, vd, n_split=3, scale=-0.1)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=-0.1)
    assert_parity(o, lse, ro, rl, "bf16", f"split scale=-0.1 d={d}")
    q, k, v = make_qkv(1, 2, 100, 333, d, "f16", seed=590 + d)
    o, lse = fwd_general(q.to(DEV), k.to(DEV), v.to(DEV), mask=ATTN_MASK_CAUSAL_BOTTOM_RIGHT,
                         scale=-0.1)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=True, scale=-0.1, bottom_right=True)
    assert_parity(o, lse, ro, rl, "f16", f"bottom-right scale=-0.1 d={d}")
