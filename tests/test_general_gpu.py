"""GPU parity of the general-layout forward (attn_fwd_general) against the fp64 oracle.

Layouts only change addressing, so results are compared with the oracle on
dense copies of the same values; grouped key/value heads are compared with the
oracle on K/V whose heads are repeated explicitly; the bottom-right causal
mask is compared with the oracle's bottom-right reading.
"""

import math

import pytest
import torch

import oracle
from exact_attention_53_gb300 import attn_get_device_status, fwd, fwd_general
from exact_attention_53_gb300.binding import (ATTN_MASK_CAUSAL, ATTN_MASK_CAUSAL_BOTTOM_RIGHT,
                                              ATTN_MASK_NONE, AttnError)
from exact_attention_53_gb300.workloads import WORKLOADS, make_qkv, workload_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_53_gb300.build import build
    build()
    yield
    attn_get_device_status()


def _oracle(q, k, v, mask, scale):
    """q [B,H,S_q,d], k/v [B,H_kv,S_k,d] (CPU, any strides) -> oracle (o, lse)."""
    group = q.shape[1] // k.shape[1]
    k = k.contiguous().repeat_interleave(group, dim=1)
    v = v.contiguous().repeat_interleave(group, dim=1)
    return oracle.attention_forward(q.contiguous(), k, v, causal=mask != ATTN_MASK_NONE,
                                    scale=scale, bottom_right=mask == ATTN_MASK_CAUSAL_BOTTOM_RIGHT)


def _bshd(t):
    """A [B,H,S,d] tensor copied into [B,S,H,d] storage, returned as a [B,H,S,d] view."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


@pytest.mark.parametrize("mask", [ATTN_MASK_NONE, ATTN_MASK_CAUSAL, ATTN_MASK_CAUSAL_BOTTOM_RIGHT],
                         ids=["full", "causal", "bottom_right"])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (8, 2), (6, 1)], ids=["mha", "gqa4", "mqa"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_bshd_gqa_masks(d, dtype, H, H_kv, mask):
    B, S_q, S_k = 2, 200, 333
    q, _, _ = make_qkv(B, H, S_q, 1, d, dtype, seed=d + H * 7 + mask)
    _, k, v = make_qkv(B, H_kv, 1, S_k, d, dtype, seed=d + H_kv * 11 + mask)
    scale = 1 / math.sqrt(d)
    qd, kd, vd = _bshd(q.to(DEV)), _bshd(k.to(DEV)), _bshd(v.to(DEV))
    o = _bshd(torch.zeros((B, H, S_q, d), dtype=q.dtype, device=DEV))
    o, lse = fwd_general(qd, kd, vd, mask=mask, scale=scale, out=o)
    torch.cuda.synchronize()
    ro, rl = _oracle(q, k, v, mask, scale)
    assert_parity(o, lse, ro, rl, dtype, f"d={d} {dtype} H={H} H_kv={H_kv} mask={mask}")


@pytest.mark.parametrize("S_q,S_k", [(1, 700), (100, 333), (256, 640), (129, 129), (300, 2000)])
def test_bottom_right_shapes(S_q, S_k):
    q, k, v = make_qkv(1, 2, S_q, S_k, 128, "bf16", seed=S_q + S_k)
    o, lse = fwd_general(q.to(DEV), k.to(DEV), v.to(DEV), mask=ATTN_MASK_CAUSAL_BOTTOM_RIGHT)
    torch.cuda.synchronize()
    ro, rl = _oracle(q, k, v, ATTN_MASK_CAUSAL_BOTTOM_RIGHT, 1 / math.sqrt(128))
    assert_parity(o, lse, ro, rl, "bf16", f"bottom-right {S_q}x{S_k}")


def test_packed_qkv_views():
    """q, k, v as views of one [B, S, 3, H, d] buffer; o written into a [B, S, H, d] buffer."""
    B, S, H, d = 2, 300, 4, 128
    qkv = torch.randn((B, S, 3, H, d), generator=torch.Generator().manual_seed(41)).to(torch.bfloat16)
    qkv_d = qkv.to(DEV)
    q, k, v = (qkv_d[:, :, i].transpose(1, 2) for i in range(3))
    out = torch.zeros((B, S, H, d), dtype=torch.bfloat16, device=DEV)
    o, lse = fwd_general(q, k, v, mask=ATTN_MASK_CAUSAL, out=out.transpose(1, 2))
    torch.cuda.synchronize()
    qc, kc, vc = (qkv[:, :, i].transpose(1, 2) for i in range(3))
    ro, rl = _oracle(qc, kc, vc, ATTN_MASK_CAUSAL, 1 / math.sqrt(d))
    assert_parity(out.transpose(1, 2), lse, ro, rl, "bf16", "packed qkv")


def test_general_matches_dense_path_bitwise_at_full_size():
    """c3 in [B, S, H, d] storage gives exactly the dense entry point's result."""
    w = WORKLOADS["c3"]
    q, k, v = (t.to(DEV) for t in workload_qkv(w))
    for causal in (False, True):
        o1, l1 = fwd(q, k, v, causal=causal, scale=w.scale)
        o2, l2 = fwd_general(_bshd(q), _bshd(k), _bshd(v),
                             mask=ATTN_MASK_CAUSAL if causal else ATTN_MASK_NONE, scale=w.scale,
                             out=_bshd(torch.empty_like(q)))
        torch.cuda.synchronize()
        assert torch.equal(o1, o2.contiguous()) and torch.equal(l1, l2)


def test_gqa_matches_repeated_heads_bitwise():
    """Grouped heads read the same K/V as explicitly repeated heads would."""
    q, _, _ = make_qkv(1, 8, 500, 1, 128, "bf16", seed=42)
    _, k, v = make_qkv(1, 2, 1, 700, 128, "bf16", seed=43)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = fwd_general(qd, kd, vd, mask=ATTN_MASK_CAUSAL)
    o2, l2 = fwd(qd, kd.repeat_interleave(4, dim=1).contiguous(),
                 vd.repeat_interleave(4, dim=1).contiguous(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bottom_right_rejects_longer_queries_on_gpu():
    q, k, v = make_qkv(1, 1, 300, 200, 64, "bf16", seed=44)
    with pytest.raises(AttnError, match="S_q <= S_k"):
        fwd_general(q.to(DEV), k.to(DEV), v.to(DEV), mask=ATTN_MASK_CAUSAL_BOTTOM_RIGHT)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mode", ["full", "causal", "split"])
def test_forward_writes_only_inside_the_output_view(d, mode):
    """O as a slice of a larger buffer (64 more columns per row, 7 more rows per head): the
    padding keeps its sentinel, and O and LSE equal the dense entry point's bit for bit."""
    from exact_attention_53_gb300 import fwd_splitkv, fwd_splitkv_general
    B, H = 1, 3
    S_q, S_k = (5, 3000) if mode == "split" else (333, 333)
    q, k, v = make_qkv(B, H, S_q, S_k, d, "bf16", seed=80 + d)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    sentinel = -123.0
    buf = torch.full((B, H, S_q + 7, d + 64), sentinel, dtype=torch.bfloat16, device=DEV)
    view = buf[:, :, :S_q, :d]
    if mode == "split":
        ro, rl = fwd_splitkv(qd, kd, vd, n_split=3)
        o, lse = fwd_splitkv_general(qd, kd, vd, n_split=3, out=view)
    else:
        causal = mode == "causal"
        ro, rl = fwd(qd, kd, vd, causal=causal)
        o, lse = fwd_general(qd, kd, vd, mask=ATTN_MASK_CAUSAL if causal else ATTN_MASK_NONE,
                             out=view)
    torch.cuda.synchronize()
    assert torch.equal(view, ro) and torch.equal(lse, rl)
    assert (buf[:, :, :, d:] == sentinel).all(), "written past the view's columns"
    assert (buf[:, :, S_q:, :] == sentinel).all(), "written past the view's rows"
