"""fp64 CPU oracle for the exact scaled-dot-product attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
this module.  The CUDA product path never routes through it, and it shares no
code, constants or helpers with ``exact_attention_53_gb300/csrc``.

What it computes
----------------
Source: oxicuda-dnn 0.1.8, ``src/attn/flash_attn/hopper.rs``, doc comment of
``FlashAttention3Plan::generate_forward``.  Per KV tile the consumer warps form
``S = Q·Kᵀ``, keep a running row maximum ``m`` and running row sum ``l`` (online
softmax), mask future token positions when causal, accumulate
``O_acc += P·V``, and after the last tile write ``O = O_acc / l`` and the
log-sum-exp ``m + log(l)``.  The online recurrence is an exact reordering of the
plain softmax (the running max only changes which constant is subtracted
before ``exp``), so this oracle is the plain definition written out:

    S      = scale · Q · Kᵀ                      (S_q × S_k, one (b, h) at a time)
    S[i,j] = −∞  for j > i                        (causal only; top-left aligned)
    m_i    = max_j S[i,j]
    P      = exp(S − m_i)          l_i = Σ_j P[i,j]
    O      = (P / l) · V           LSE_i = m_i + ln(l_i)

Readings taken where the page is silent:
  * "zero out future token positions" is read as the masked logit being −∞
    (its probability is zero), not the score being set to 0.
  * causal alignment is top-left: key j is visible to query i iff j ≤ i.
    ``bottom_right=True`` (an option the page does not have, for S_q ≤ S_k)
    aligns the last query with the last key instead: j ≤ i + (S_k − S_q).
  * the log-sum-exp is the natural log and includes the scale:
    LSE_i = ln Σ_j exp(scale · q_i · k_j).
  * the scale is any finite number (the page's ``sm_scale`` is a plain f32):
    zero gives uniform weights, a negative scale favours the keys least
    aligned with the query.
  * inputs are the fp16/bf16 values exactly as stored, widened to fp64; the
    oracle does not round P or O to the input dtype.

Rows are processed in blocks of at most ``row_block`` queries, each block
against the full key length; this only bounds memory, every row is computed
independently in the same way.
"""

from __future__ import annotations

import numpy as np

__all__ = ["attention_forward", "attention_rows", "attention_probs"]


def _as_f64(x) -> np.ndarray:
    """Widen an array (numpy, or anything with ``__array__``) to float64."""
    if hasattr(x, "detach"):  # a torch tensor: widen through float32, exact for f16/bf16
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def _head(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: np.ndarray,
          causal: bool, scale: float, offset: int = 0):
    """Attention for the query rows ``rows`` of one (b, h): returns (o, lse).

    Under ``causal`` key j is visible to query i iff j <= i + offset.
    """
    s = scale * (q[rows] @ k.T)                       # [R, S_k]
    if causal:
        keys = np.arange(k.shape[0])
        s = np.where(keys[None, :] > rows[:, None] + offset, -np.inf, s)
    m = s.max(axis=1, keepdims=True)                  # row maximum
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)                  # row sum
    o = (p @ v) / l
    lse = m[:, 0] + np.log(l[:, 0])
    return o, lse


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None,
                      row_block: int = 512, bottom_right: bool = False):
    """O and LSE for ``q [B,H,S_q,d]``, ``k [B,H,S_k,d]``, ``v [B,H,S_k,d_v]``.

    Returns ``(o, lse)`` as float64 arrays of shapes ``[B,H,S_q,d_v]`` and
    ``[B,H,S_q]``.  ``scale`` defaults to ``1/sqrt(d)``.  ``bottom_right``
    (with ``causal``, S_q <= S_k) shifts the mask by S_k − S_q.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, S_q, d = q.shape
    if k.shape[:2] != (B, H) or v.shape[:3] != k.shape[:3] or k.shape[3] != d:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    offset = 0
    if causal and bottom_right:
        if S_q > k.shape[2]:
            raise ValueError("bottom-right alignment needs S_q <= S_k")
        offset = k.shape[2] - S_q
    o = np.empty((B, H, S_q, v.shape[3]), dtype=np.float64)
    lse = np.empty((B, H, S_q), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, S_q, row_block):
                rows = np.arange(r0, min(r0 + row_block, S_q))
                o[b, h, rows], lse[b, h, rows] = _head(q[b, h], k[b, h], v[b, h],
                                                        rows, causal, scale, offset)
    return o, lse


def attention_rows(q_bh, k_bh, v_bh, rows, causal: bool = False,
                   scale: float | None = None, bottom_right: bool = False):
    """O and LSE for selected query ``rows`` of a single head.

    ``q_bh [S_q,d]``, ``k_bh, v_bh [S_k,d]``; returns ``(o [R,d], lse [R])``.
    Used to check full-size outputs at sampled rows.
    """
    q, k, v = _as_f64(q_bh), _as_f64(k_bh), _as_f64(v_bh)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[1])
    rows = np.asarray(rows, dtype=np.int64)
    offset = k.shape[0] - q.shape[0] if (causal and bottom_right) else 0
    return _head(q, k, v, rows, causal, scale, offset)


def attention_probs(q_bh, k_bh, causal: bool = False, scale: float | None = None):
    """The softmax matrix ``P = softmax(scale·Q·Kᵀ [+mask])`` of one head.

    Exposed so the row-sum and masking invariants can be checked directly.
    """
    q, k = _as_f64(q_bh), _as_f64(k_bh)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[1])
    s = scale * (q @ k.T)
    if causal:
        i = np.arange(q.shape[0])[:, None]
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > i, -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    return p / p.sum(axis=1, keepdims=True)
