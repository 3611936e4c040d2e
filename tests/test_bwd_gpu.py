"""GPU parity of the attention backward (through the C ABI) against the fp64 oracle.

Tolerance (derived from the arithmetic; the pages state none for gradients).
The kernels read O and LSE from the GPU forward, round P and dS to the input
dtype for the tensor-core products, accumulate in fp32 and round dQ, dK, dV
to the dtype.  With u = 2⁻⁸ (bf16) or 2⁻¹¹ (f16), twice the unit roundoff,
each element must satisfy |Δ| ≤ 2·bound + 1e-6·max|ref| where

    δD_i   = 2u · Σ_c |dO_ic| · (|P|·|V|)_ic            (O as rounded by the forward)
    δdS_ij = P_ij · δD_i + u · |dS_ij|                  (dS rounded to the dtype)
    dV:  2u · (|P|ᵀ·|dO|)_jc       + u·|dV_jc|
    dK:  |scale| · (δdSᵀ·|Q|)_jc   + u·|dK_jc|
    dQ:  |scale| · (δdS·|K|)_ic    + u·|dQ_ic|

all formed in fp64 from the oracle's exact P, dS, V, dO, Q, K.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_53_gb300 import attn_get_device_status, bwd, fwd
from exact_attention_53_gb300.workloads import WORKLOADS, make_qkv, workload_qkv

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


def _check_head(got, q, k, v, do, causal, scale, dtype, what):
    """got = (dq, dk, dv) of one head as fp64 arrays; q, k, v, do the head's inputs."""
    t = oracle.backward_terms(q, k, v, do, causal=causal, scale=scale)
    u = UNIT[dtype]
    P, dS = t["P"], t["dS"]
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(do)
    dD = 2 * u * (np.abs(dO) * (np.abs(P) @ np.abs(V))).sum(axis=1)
    ddS = P * dD[:, None] + u * np.abs(dS)
    bounds = {
        "dV": 2 * u * (np.abs(P).T @ np.abs(dO)) + u * np.abs(t["dV"]),
        "dK": abs(scale) * (ddS.T @ np.abs(Q)) + u * np.abs(t["dK"]),
        "dQ": abs(scale) * (ddS @ np.abs(K)) + u * np.abs(t["dQ"]),
    }
    for name, g in zip(("dQ", "dK", "dV"), got):
        ref = t[name]
        assert np.isfinite(g).all(), f"{what}: non-finite {name}"
        tol = 2 * bounds[name] + 1e-6 * max(np.abs(ref).max(), 1e-30)
        err = np.abs(g - ref)
        if (err > tol).any():
            idx = np.unravel_index(np.argmax(err - tol), err.shape)
            raise AssertionError(f"{what}: {name} {(err > tol).sum()} elements out of tolerance; "
                                 f"worst at {idx}: gpu={g[idx]:.6g} ref={ref[idx]:.6g} "
                                 f"tol={tol[idx]:.3g} max|d|={err.max():.3g}")


def _run_bwd(q, k, v, do, causal, scale):
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    o, lse = fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return dq, dk, dv


SHAPES = [(1, 1, 1, 1), (1, 2, 17, 17), (1, 1, 64, 64), (2, 1, 127, 127), (1, 2, 128, 128),
          (1, 1, 129, 129), (1, 1, 200, 333), (1, 1, 333, 200), (1, 2, 300, 300), (1, 1, 1, 700),
          (1, 1, 700, 1)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_bwd_small_shapes(d, dtype, causal, shape):
    B, H, S_q, S_k = shape
    seed = S_q * 7907 + S_k * 37 + d + (1 if causal else 0)
    q, k, v = make_qkv(B, H, S_q, S_k, d, dtype, seed=seed)
    do = make_qkv(B, H, S_q, 1, d, dtype, seed=seed + 1)[0]
    scale = 1 / math.sqrt(d)
    dq, dk, dv = _run_bwd(q, k, v, do, causal, scale)
    for b in range(B):
        for h in range(H):
            got = (_f64(dq[b, h]), _f64(dk[b, h]), _f64(dv[b, h]))
            _check_head(got, q[b, h], k[b, h], v[b, h], do[b, h], causal, scale, dtype,
                        f"d={d} {dtype} causal={causal} {shape} head=({b},{h})")


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_bwd_negative_scale(d, dtype, causal):
    """A negative scale (the page's sm_scale is any f32): forward and backward of the same
    problem, gradients within the derived bound (with |scale| in it)."""
    B, H, S = 1, 2, 300
    q, k, v = make_qkv(B, H, S, S, d, dtype, seed=610 + d)
    do = make_qkv(B, H, S, 1, d, dtype, seed=611 + d)[0]
    dq, dk, dv = _run_bwd(q, k, v, do, causal, -0.1)
    for h in range(H):
        got = (_f64(dq[0, h]), _f64(dk[0, h]), _f64(dv[0, h]))
        _check_head(got, q[0, h], k[0, h], v[0, h], do[0, h], causal, -0.1, dtype,
                    f"scale=-0.1 d={d} {dtype} causal={causal} head={h}")


def test_bwd_c2_full():
    """The d=64, S=1024 causal workload at full size, every head."""
    w = WORKLOADS["c2"]
    q, k, v = workload_qkv(w)
    do = make_qkv(w.B, w.H, w.S_q, 1, w.d, w.dtype, seed=w.seed + 100)[0]
    dq, dk, dv = _run_bwd(q, k, v, do, True, w.scale)
    for b in range(w.B):
        for h in range(w.H):
            got = (_f64(dq[b, h]), _f64(dk[b, h]), _f64(dv[b, h]))
            _check_head(got, q[b, h], k[b, h], v[b, h], do[b, h], True, w.scale, w.dtype,
                        f"c2 head=({b},{h})")


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_c3_sampled_heads(causal):
    """The d=128, S=4096 workload at full size; three heads compared in full."""
    w = WORKLOADS["c3"]
    q, k, v = workload_qkv(w)
    do = make_qkv(w.B, w.H, w.S_q, 1, w.d, w.dtype, seed=w.seed + 100)[0]
    dq, dk, dv = _run_bwd(q, k, v, do, causal, w.scale)
    for b, h in ((0, 0), (1, 31), (1, 5)):
        got = (_f64(dq[b, h]), _f64(dk[b, h]), _f64(dv[b, h]))
        _check_head(got, q[b, h], k[b, h], v[b, h], do[b, h], causal, w.scale, w.dtype,
                    f"c3 causal={causal} head=({b},{h})")


def test_bwd_c5_sampled_heads():
    """The d=256, S=8192 workload at full size (the two-pass key side); two heads in full."""
    w = WORKLOADS["c5"]
    q, k, v = workload_qkv(w)
    do = make_qkv(w.B, w.H, w.S_q, 1, w.d, w.dtype, seed=w.seed + 100)[0]
    dq, dk, dv = _run_bwd(q, k, v, do, False, w.scale)
    for b, h in ((0, 0), (1, 7)):
        got = (_f64(dq[b, h]), _f64(dk[b, h]), _f64(dv[b, h]))
        _check_head(got, q[b, h], k[b, h], v[b, h], do[b, h], False, w.scale, w.dtype,
                    f"c5 head=({b},{h})")


@pytest.mark.parametrize("d", [128, 256])
def test_bwd_deterministic(d):
    q, k, v = make_qkv(2, 3, 500, 700, d, "bf16", seed=31)
    do = make_qkv(2, 3, 500, 1, d, "bf16", seed=32)[0]
    for causal in (False, True):
        a = _run_bwd(q, k, v, do, causal, 0.1)
        b = _run_bwd(q, k, v, do, causal, 0.1)
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_repeated_calls_stay_clean_and_identical(causal):
    """Eight back-to-back backward calls on c3: no bounded wait runs out (checked on the
    device status) and every call gives the first call's bits."""
    w = WORKLOADS["c3"]
    q, k, v = (t.to(DEV) for t in workload_qkv(w))
    do = make_qkv(w.B, w.H, w.S_q, 1, w.d, w.dtype, seed=w.seed + 100)[0].to(DEV)
    o, lse = fwd(q, k, v, causal=causal, scale=w.scale)
    first = bwd(q, k, v, o, lse, do, causal=causal, scale=w.scale)
    rest = [bwd(q, k, v, o, lse, do, causal=causal, scale=w.scale) for _ in range(7)]
    torch.cuda.synchronize()
    attn_get_device_status()
    for grads in rest:
        for x, y in zip(grads, first):
            assert torch.equal(x, y)


def test_bwd_scale_zero():
    q, k, v = make_qkv(1, 2, 150, 190, 64, "f16", seed=33)
    do = make_qkv(1, 2, 150, 1, 64, "f16", seed=34)[0]
    dq, dk, dv = _run_bwd(q, k, v, do, False, 0.0)
    assert torch.all(dq == 0) and torch.all(dk == 0)
    for h in range(2):
        _check_head((_f64(dq[0, h]), _f64(dk[0, h]), _f64(dv[0, h])), q[0, h], k[0, h], v[0, h],
                    do[0, h], False, 0.0, "f16", f"scale 0 head {h}")


def test_bwd_key_gradients_sum_to_zero():
    """Σ_j dK_j = 0 per head (softmax shift invariance), within the bf16 bound."""
    q, k, v = make_qkv(1, 2, 512, 512, 128, "bf16", seed=35)
    do = make_qkv(1, 2, 512, 1, 128, "bf16", seed=36)[0]
    for causal in (False, True):
        _, dk, _ = _run_bwd(q, k, v, do, causal, 1 / math.sqrt(128))
        s = dk.float().sum(dim=2)
        scale = dk.float().abs().sum(dim=2)
        assert (s.abs() <= 0.02 * scale + 1e-3).all()


def _bwd_into(q, k, v, o, lse, do, dq, dk, dv, ws, causal, scale):
    from exact_attention_53_gb300 import attn_bwd
    B, H, S_q, d = q.shape
    attn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, S_q, k.shape[2], d, int(causal), scale, 1, ws,
             ws.numel())


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_result_ordered_on_callers_stream(causal):
    """dQ is computed on a helper stream; work queued on the caller's stream after the call
    must see all three gradients complete (the call joins the helper stream back)."""
    from exact_attention_53_gb300 import attn_bwd_workspace_size
    q, k, v = (t.to(DEV) for t in make_qkv(2, 8, 1024, 1024, 128, "bf16", seed=37))
    do = make_qkv(2, 8, 1024, 1, 128, "bf16", seed=38)[0].to(DEV)
    scale = 1 / math.sqrt(128)
    o, lse = fwd(q, k, v, causal=causal, scale=scale)
    ws = torch.empty(attn_bwd_workspace_size(2, 8, 1024, 1024, 128, 1), dtype=torch.uint8,
                     device=DEV)
    ref = bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(5):
            dq, dk, dv = (torch.zeros_like(t) for t in (q, k, v))
            _bwd_into(q, k, v, o, lse, do, dq, dk, dv, ws, causal, scale)
            copies = [t.clone() for t in (dq, dk, dv)]     # queued right behind the call
            s.synchronize()
            for x, y in zip(copies, ref):
                assert torch.equal(x, y)


def test_bwd_captures_into_a_cuda_graph():
    """A stream capture of the call takes the helper stream in with it; replays give the
    eager result bit for bit."""
    from exact_attention_53_gb300 import attn_bwd_workspace_size
    q, k, v = (t.to(DEV) for t in make_qkv(1, 4, 700, 900, 64, "f16", seed=39))
    do = make_qkv(1, 4, 700, 1, 64, "f16", seed=40)[0].to(DEV)
    o, lse = fwd(q, k, v, scale=0.125)
    ws = torch.empty(attn_bwd_workspace_size(1, 4, 700, 900, 64, 0), dtype=torch.uint8,
                     device=DEV)
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    from exact_attention_53_gb300 import attn_bwd

    def call():
        attn_bwd(q, k, v, o, lse, do, dq, dk, dv, 1, 4, 700, 900, 64, 0, 0.125, 0, ws, ws.numel())

    call()                                              # eager (creates the helper stream)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    with torch.cuda.graph(g, stream=s):
        call()
    for _ in range(3):
        for t in (dq, dk, dv):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for x, y in zip((dq, dk, dv), ref):
            assert torch.equal(x, y)
