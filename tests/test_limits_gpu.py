"""GPU parity at the size limits the library accepts.

S_k = 2^22 keys (the largest sequence length attn_fwd accepts) for two query
rows, through the one-pass kernel (a single work unit walks all 32768 key
tiles), the split-KV path and the bottom-right causal mask; and a problem with
many more work units than SMs (every persistent CTA loops over ~50 units).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_53_gb300 import attn_get_device_status, fwd, fwd_general, fwd_splitkv
from exact_attention_53_gb300.binding import ATTN_MASK_CAUSAL_BOTTOM_RIGHT
from exact_attention_53_gb300.workloads import make_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_53_gb300.build import build
    build()
    yield
    attn_get_device_status()


@pytest.fixture(scope="module")
def longest():
    S_k = 1 << 22
    q, k, v = make_qkv(1, 1, 2, S_k, 64, "bf16", seed=61)
    return q, k, v, (q.to(DEV), k.to(DEV), v.to(DEV))


def test_longest_keys_one_pass_and_split(longest):
    q, k, v, (qd, kd, vd) = longest
    scale = 1 / 8
    o1, l1 = fwd(qd, kd, vd, scale=scale)
    o2, l2 = fwd_splitkv(qd, kd, vd, n_split=0, scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_rows(q[0, 0], k[0, 0], v[0, 0], np.arange(2), scale=scale)
    assert_parity(o1[0, 0], l1[0, 0], ro, rl, "bf16", "S_k=2^22 one-pass")
    assert_parity(o2[0, 0], l2[0, 0], ro, rl, "bf16", "S_k=2^22 split-KV")


def test_longest_keys_bottom_right(longest):
    q, k, v, (qd, kd, vd) = longest
    o, lse = fwd_general(qd, kd, vd, mask=ATTN_MASK_CAUSAL_BOTTOM_RIGHT, scale=1 / 8)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_rows(q[0, 0], k[0, 0], v[0, 0], np.arange(2), causal=True,
                                   scale=1 / 8, bottom_right=True)
    assert_parity(o[0, 0], lse[0, 0], ro, rl, "bf16", "S_k=2^22 bottom-right")


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_many_more_units_than_sms(causal):
    """64·32 heads of 300 rows: 2048 one-block units for 152 persistent CTAs."""
    B, H, S, d = 64, 32, 300, 64
    q, k, v = make_qkv(B, H, S, S, d, "f16", seed=62)
    o, lse = fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    rng = np.random.default_rng(63)
    for b, h in {(0, 0), (B - 1, H - 1), *((int(x), int(y)) for x, y in rng.integers(0, (B, H), (6, 2)))}:
        ro, rl = oracle.attention_forward(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                          v[b:b + 1, h:h + 1], causal=causal,
                                          scale=1 / math.sqrt(d))
        assert_parity(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], ro, rl, "f16",
                      f"head ({b},{h}) causal={causal}")


def test_grid_beyond_65535_units():
    """66560 one-block units: a grid far past 65535 CTAs, all but about one per SM taken over
    through the work queue.  Every output row must be written (O starts as NaN), and sampled
    heads, the first and the last among them, match the oracle.  Heads of different batches
    get different V (a per-batch offset), so a unit written to the wrong place shows up."""
    B, H, S, d = 512, 130, 128, 64
    q1, k1, v1 = (t.to(DEV) for t in make_qkv(1, H, S, S, d, "bf16", seed=64))
    shift = (torch.arange(B, device=DEV, dtype=torch.float32) / B).view(B, 1, 1, 1)
    q = q1.expand(B, -1, -1, -1).contiguous()
    k = k1.expand(B, -1, -1, -1).contiguous()
    v = (v1.float() + shift).to(torch.bfloat16)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=DEV)
    o, lse = fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all().item() and torch.isfinite(lse).all().item()
    rng = np.random.default_rng(65)
    picks = {(0, 0), (B - 1, H - 1), *((int(x), int(y)) for x, y in rng.integers(0, (B, H), (6, 2)))}
    for b, h in picks:
        qc, kc, vc = (t[b:b + 1, h:h + 1].cpu() for t in (q, k, v))
        ro, rl = oracle.attention_forward(qc, kc, vc, causal=True, scale=1 / math.sqrt(d))
        assert_parity(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], ro, rl, "bf16",
                      f"head ({b},{h}) of {B * H}")
