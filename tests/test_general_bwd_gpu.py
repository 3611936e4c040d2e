"""GPU parity of the general-layout backward (attn_bwd_general) against the fp64 oracle.

Strided layouts change only addressing.  With grouped key/value heads the
gradient of a shared K/V head is the sum over the query heads that read it
(the chain rule through the head repetition), so the reference and its error
bound are the oracle's per-query-head dK, dV (and bounds) summed over each
group.  The per-element bound is the one derived in test_bwd_gpu.py.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_53_gb300 import attn_get_device_status, bwd, bwd_general, fwd, fwd_general
from exact_attention_53_gb300.binding import (ATTN_MASK_CAUSAL, ATTN_MASK_CAUSAL_BOTTOM_RIGHT,
                                              ATTN_MASK_NONE)
from exact_attention_53_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
UNIT = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_53_gb300.build import build
    build()
    yield
    attn_get_device_status()


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _bshd(t):
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _reference(q, k, v, do, mask, scale, dtype):
    """Per-(b, h) oracle terms -> (dq, dk, dv) references and their bounds, K/V per kv head."""
    B, H, S_q, d = q.shape
    H_kv, S_k = k.shape[1], k.shape[2]
    group = H // H_kv
    u = UNIT[dtype]
    ref = {n: np.zeros(s) for n, s in (("dQ", (B, H, S_q, d)), ("dK", (B, H_kv, S_k, d)),
                                       ("dV", (B, H_kv, S_k, d)))}
    bnd = {n: np.zeros_like(r) for n, r in ref.items()}
    for b in range(B):
        for h in range(H):
            hk = h // group
            t = oracle.backward_terms(q[b, h], k[b, hk], v[b, hk], do[b, h],
                                      causal=mask != ATTN_MASK_NONE, scale=scale,
                                      bottom_right=mask == ATTN_MASK_CAUSAL_BOTTOM_RIGHT)
            P, dS = t["P"], t["dS"]
            Q, K, V, dO = _f64(q[b, h]), _f64(k[b, hk]), _f64(v[b, hk]), _f64(do[b, h])
            dD = 2 * u * (np.abs(dO) * (np.abs(P) @ np.abs(V))).sum(axis=1)
            ddS = P * dD[:, None] + u * np.abs(dS)
            ref["dQ"][b, h] = t["dQ"]
            ref["dK"][b, hk] += t["dK"]
            ref["dV"][b, hk] += t["dV"]
            bnd["dQ"][b, h] = scale * (ddS @ np.abs(K)) + u * np.abs(t["dQ"])
            bnd["dK"][b, hk] += scale * (ddS.T @ np.abs(Q)) + u * np.abs(t["dK"])
            bnd["dV"][b, hk] += 2 * u * (np.abs(P).T @ np.abs(dO)) + u * np.abs(t["dV"])
    return ref, bnd


def _check(got, ref, bnd, what):
    for name, g in zip(("dQ", "dK", "dV"), got):
        g = _f64(g)
        r = ref[name]
        tol = 2 * bnd[name] + 1e-6 * max(np.abs(r).max(), 1e-30)
        err = np.abs(g - r)
        assert np.isfinite(g).all(), f"{what}: non-finite {name}"
        if (err > tol).any():
            idx = np.unravel_index(np.argmax(err - tol), err.shape)
            raise AssertionError(f"{what}: {name} {(err > tol).sum()} out of tolerance; worst at "
                                 f"{idx}: gpu={g[idx]:.6g} ref={r[idx]:.6g} tol={tol[idx]:.3g}")


@pytest.mark.parametrize("mask", [ATTN_MASK_NONE, ATTN_MASK_CAUSAL, ATTN_MASK_CAUSAL_BOTTOM_RIGHT],
                         ids=["full", "causal", "bottom_right"])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (8, 2), (6, 1)], ids=["mha", "gqa4", "mqa"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_bwd_bshd_gqa_masks(d, dtype, H, H_kv, mask):
    B, S_q, S_k = 1, 200, 333
    q, _, _ = make_qkv(B, H, S_q, 1, d, dtype, seed=3 * d + H + mask)
    _, k, v = make_qkv(B, H_kv, 1, S_k, d, dtype, seed=5 * d + H_kv + mask)
    do = make_qkv(B, H, S_q, 1, d, dtype, seed=7 * d + H + mask)[0]
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = _bshd(q.to(DEV)), _bshd(k.to(DEV)), _bshd(v.to(DEV)), _bshd(do.to(DEV))
    o, lse = fwd_general(qd, kd, vd, mask=mask, scale=scale, out=_bshd(torch.empty_like(qd)))
    grads = bwd_general(qd, kd, vd, o, lse, dod, mask=mask, scale=scale,
                        dq=_bshd(torch.empty_like(qd)), dk=_bshd(torch.empty_like(kd)),
                        dv=_bshd(torch.empty_like(vd)))
    torch.cuda.synchronize()
    ref, bnd = _reference(q, k, v, do, mask, scale, dtype)
    _check(grads, ref, bnd, f"d={d} {dtype} H={H} H_kv={H_kv} mask={mask}")


@pytest.mark.parametrize("S_q,S_k", [(1, 300), (64, 500), (130, 129 + 260)])
def test_bwd_bottom_right_shapes(S_q, S_k):
    q, k, v = make_qkv(1, 2, S_q, S_k, 128, "bf16", seed=S_q * 3 + S_k)
    do = make_qkv(1, 2, S_q, 1, 128, "bf16", seed=S_q * 5 + S_k)[0]
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    mask = ATTN_MASK_CAUSAL_BOTTOM_RIGHT
    o, lse = fwd_general(qd, kd, vd, mask=mask)
    grads = bwd_general(qd, kd, vd, o, lse, dod, mask=mask)
    torch.cuda.synchronize()
    ref, bnd = _reference(q, k, v, do, mask, 1 / math.sqrt(128), "bf16")
    _check(grads, ref, bnd, f"bottom-right {S_q}x{S_k}")


def test_bwd_general_matches_dense_bitwise():
    """[B, S, H, d] storage gives exactly the dense entry point's gradients."""
    q, k, v = make_qkv(2, 4, 700, 700, 128, "bf16", seed=51)
    do = make_qkv(2, 4, 700, 1, 128, "bf16", seed=52)[0]
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    for causal in (False, True):
        o, lse = fwd(qd, kd, vd, causal=causal)
        a = bwd(qd, kd, vd, o, lse, dod, causal=causal)
        b = bwd_general(_bshd(qd), _bshd(kd), _bshd(vd), _bshd(o), lse, _bshd(dod),
                        mask=ATTN_MASK_CAUSAL if causal else ATTN_MASK_NONE,
                        dq=_bshd(torch.empty_like(qd)), dk=_bshd(torch.empty_like(kd)),
                        dv=_bshd(torch.empty_like(vd)))
        torch.cuda.synchronize()
        for x, y in zip(a, b):
            assert torch.equal(x, y.contiguous())


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_writes_only_inside_the_gradient_views(d, causal):
    """dQ, dK, dV as slices of larger buffers (64 more columns per row, 7 more rows per head):
    the padding keeps its sentinel, so the tile stores never write past a view's columns or
    its S rows, and the gradients equal the dense entry point's bit for bit."""
    B, H, S = 1, 3, 333
    q, k, v = make_qkv(B, H, S, S, d, "bf16", seed=60 + d)
    do = make_qkv(B, H, S, 1, d, "bf16", seed=61 + d)[0]
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    o, lse = fwd(qd, kd, vd, causal=causal)
    ref = bwd(qd, kd, vd, o, lse, dod, causal=causal)
    sentinel = -123.0
    bufs = [torch.full((B, H, S + 7, d + 64), sentinel, dtype=torch.bfloat16, device=DEV)
            for _ in range(3)]
    views = [bb[:, :, :S, :d] for bb in bufs]
    bwd_general(qd, kd, vd, o, lse, dod, mask=ATTN_MASK_CAUSAL if causal else ATTN_MASK_NONE,
                dq=views[0], dk=views[1], dv=views[2])
    torch.cuda.synchronize()
    for name, bb, view, want in zip(("dq", "dk", "dv"), bufs, views, ref):
        assert torch.equal(view, want), f"{name}: differs from the dense call"
        assert (bb[:, :, :, d:] == sentinel).all(), f"{name}: written past its columns"
        assert (bb[:, :, S:, :] == sentinel).all(), f"{name}: written past its rows"
