"""fp64 CPU oracle for the exact attention backward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
this module.  It shares no code with ``exact_attention_53_gb300/csrc``.

What it computes
----------------
Source: oxicuda-dnn 0.1.8, ``src/attn/flash_attn/hopper.rs``, doc comment of
``FlashAttention3Plan::generate_backward``.  With the forward's probabilities
recomputed from its saved log-sum-exp, the page lists the gradient steps

    dV = Pᵀ·dO          dP = dO·Vᵀ
    dS = P ∘ (dP − D)   with D_i = Σ_j dP_ij P_ij  (the page also writes it as
                        rowsum(dO ∘ O); the two are equal because O_i = Σ_j P_ij v_j)
    dQ = dS·K           dK = dSᵀ·Q

For the forward O = softmax(scale·Q·Kᵀ [+ mask])·V these are the exact
gradients of Σ O ∘ dO, with the scale the page passes as ``sm_scale`` applied
to dQ and dK (the chain rule through scale·Q·Kᵀ); the page's listing leaves it
implicit.  This oracle is that plain definition, one (b, h) at a time, with
P, O and D formed exactly in fp64 (not read back from a rounded forward):

    P  = softmax_rows(scale·Q·Kᵀ, masked)      O = P·V       D_i = Σ_c dO_ic O_ic
    dV = Pᵀ·dO      dP = dO·Vᵀ      dS = P ∘ (dP − D)
    dQ = scale·dS·K      dK = scale·dSᵀ·Q

Readings where the page is silent: masking and its top-left alignment as in the
forward oracle (``bottom_right`` shifts it by S_k − S_q, as there); D computed
as rowsum(dO ∘ O); the scale applied to dQ and dK.
"""

from __future__ import annotations

import numpy as np

from .attention import _as_f64

__all__ = ["attention_backward", "backward_terms"]


def backward_terms(q_bh, k_bh, v_bh, do_bh, causal: bool = False, scale: float | None = None,
                   bottom_right: bool = False):
    """Every intermediate of one head's backward: P, O, D, dP, dS, dQ, dK, dV (fp64).

    ``q_bh [S_q,d]``, ``k_bh [S_k,d]``, ``v_bh [S_k,d_v]``, ``do_bh [S_q,d_v]``.
    """
    q, k, v, do = _as_f64(q_bh), _as_f64(k_bh), _as_f64(v_bh), _as_f64(do_bh)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[1])
    s = scale * (q @ k.T)
    if causal:
        offset = k.shape[0] - q.shape[0] if bottom_right else 0
        i = np.arange(q.shape[0])[:, None]
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > i + offset, -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    p = e / e.sum(axis=1, keepdims=True)        # masked entries are exactly 0
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    dd = (do * o).sum(axis=1)                   # D_i = rowsum(dO ∘ O)
    ds = p * (dp - dd[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return {"P": p, "O": o, "D": dd, "dP": dp, "dS": ds, "dQ": dq, "dK": dk, "dV": dv}


def attention_backward(q, k, v, do, causal: bool = False, scale: float | None = None,
                       bottom_right: bool = False):
    """dQ, dK, dV (fp64) of Σ O∘dO for ``q [B,H,S_q,d]``, ``k, v [B,H,S_k,d]``, ``do [B,H,S_q,d]``."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    B, H, S_q, d = q.shape
    if k.shape[:2] != (B, H) or v.shape[:3] != k.shape[:3] or do.shape[:3] != q.shape[:3]:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape} do{do.shape}")
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    for b in range(B):
        for h in range(H):
            t = backward_terms(q[b, h], k[b, h], v[b, h], do[b, h], causal, scale, bottom_right)
            dq[b, h], dk[b, h], dv[b, h] = t["dQ"], t["dK"], t["dV"]
    return dq, dk, dv
