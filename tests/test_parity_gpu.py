"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small shapes are compared element by element over every output; the five
named workloads run at full size in the launch configuration the benchmark
uses and are compared on every row of every head, plus properties that hold
at any size (finiteness, LSE bounds).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_53_gb300 import (AttnError, attn_fwd, attn_fwd_host, attn_get_device_status,
                                      fwd)
from exact_attention_53_gb300.binding import ATTN_DTYPE_BF16, ATTN_DTYPE_F16
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


def _run(q, k, v, causal, scale):
    o, lse = fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse


# (B, H, S_q, S_k): single element, ragged tails on either side of one and two
# 128-row tiles, S_q != S_k both ways, odd B·H, one query against many keys.
SHAPES = [(1, 1, 1, 1), (1, 2, 17, 17), (2, 1, 127, 127), (1, 3, 129, 129), (1, 2, 300, 300),
          (1, 1, 200, 333), (1, 1, 333, 200), (1, 1, 256, 256), (3, 1, 64, 520), (1, 1, 1, 700)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_small_shapes(d, dtype, causal, shape):
    B, H, S_q, S_k = shape
    q, k, v = make_qkv(B, H, S_q, S_k, d, dtype, seed=S_q * 7919 + S_k * 31 + d)
    scale = 1 / math.sqrt(d)
    o, lse = _run(q, k, v, causal, scale)
    ro, rl = oracle.attention_forward(q, k, v, causal=causal, scale=scale)
    assert_parity(o, lse, ro, rl, dtype, f"d={d} {dtype} causal={causal} {shape}")


def _full_size(name, causal):
    """A named workload at full size in the benchmark's launch configuration, every row of
    every head compared with the oracle (one head at a time, to bound host memory)."""
    w = WORKLOADS[name]
    q, k, v = workload_qkv(w)
    o, lse = _run(q, k, v, causal, w.scale)
    o_cpu, lse_cpu = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o_cpu).all() and np.isfinite(lse_cpu).all()
    for b in range(w.B):
        for h in range(w.H):
            ro, rl = oracle.attention_forward(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                              v[b:b + 1, h:h + 1], causal=causal, scale=w.scale)
            assert_parity(o_cpu[b, h], lse_cpu[b, h], ro[0, 0], rl[0, 0], w.dtype,
                          f"{name} causal={causal} head=({b},{h})")


def test_c1_full():
    _full_size("c1", False)


def test_c2_full():
    _full_size("c2", True)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_c3_every_head(causal):
    _full_size("c3", causal)


def test_c4_every_head():
    _full_size("c4", True)


def test_c5_every_head():
    _full_size("c5", False)


def test_lse_bounds_at_full_size():
    """max_j S_ij <= LSE_i <= max_j S_ij + ln(#visible keys), every row of c3 causal."""
    w = WORKLOADS["c3"]
    q, k, v = workload_qkv(w)
    qd, kd = q.to(DEV), k.to(DEV)
    _, lse = fwd(qd, kd, v.to(DEV), causal=True, scale=w.scale)
    b, h = 1, 7
    s = (qd[b, h].float() @ kd[b, h].float().T) * w.scale
    s = s.masked_fill(torch.ones_like(s, dtype=torch.bool).triu(1), float("-inf"))
    mx = s.max(dim=1).values
    n = torch.arange(1, w.S_q + 1, device=DEV, dtype=torch.float32)
    assert (lse[b, h] >= mx - 1e-3).all()
    assert (lse[b, h] <= mx + torch.log(n) + 1e-3).all()


def test_deterministic():
    q, k, v = make_qkv(2, 4, 777, 777, 128, "bf16", seed=5)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    for causal in (False, True):
        o1, l1 = fwd(qd, kd, vd, causal=causal)
        o2, l2 = fwd(qd, kd, vd, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name,causal", [("c3", False), ("c3", True), ("c2", True), ("c5", False)],
                         ids=["c3-full", "c3-causal", "c2", "c5"])
def test_repeated_launches_stay_clean_and_identical(name, causal):
    """Twenty back-to-back launches of a workload: no bounded wait runs out in any of them (a
    handoff race that only some launches hit would show here) and every launch gives the
    first one's bits."""
    w = WORKLOADS[name]
    q, k, v = (t.to(DEV) for t in workload_qkv(w))
    o0, l0 = fwd(q, k, v, causal=causal, scale=w.scale)
    outs = [fwd(q, k, v, causal=causal, scale=w.scale) for _ in range(19)]
    torch.cuda.synchronize()
    attn_get_device_status()                 # raises AttnError on a timeout
    for o, lse in outs:
        assert torch.equal(o, o0) and torch.equal(lse, l0)


def test_scale_zero_gives_mean_of_values():
    q, k, v = make_qkv(1, 2, 150, 150, 64, "f16", seed=11)
    for causal in (False, True):
        o, lse = _run(q, k, v, causal, 0.0)
        ro, rl = oracle.attention_forward(q, k, v, causal=causal, scale=0.0)
        assert_parity(o, lse, ro, rl, "f16", f"scale=0 causal={causal}")


def test_constant_values():
    q, k, _ = make_qkv(1, 1, 260, 260, 128, "bf16", seed=12)
    v = torch.full((1, 1, 260, 128), 0.375, dtype=torch.bfloat16)
    for causal in (False, True):
        o, _ = _run(q, k, v, causal, 1 / math.sqrt(128))
        assert torch.all(o.float() == 0.375)


def test_large_logits_rescaling():
    """Logits growing along the key axis force the running maximum up tile after tile."""
    S, d = 1024, 128
    q, k, v = make_qkv(1, 2, S, S, d, "bf16", seed=13)
    ramp = torch.linspace(0, 6, S).view(1, 1, S, 1)
    k = (k.float() * 0.2 + ramp * q.float().mean(dim=2, keepdim=True)).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = _run(q, k, v, causal, 1.0)
        ro, rl = oracle.attention_forward(q, k, v, causal=causal, scale=1.0)
        assert_parity(o, lse, ro, rl, "bf16", f"ramped logits causal={causal}")


def test_outputs_stay_in_bounds():
    """Nothing is written outside O and LSE (canaries on both sides)."""
    B, H, S, d = 1, 3, 300, 128
    q, k, v = make_qkv(B, H, S, S, d, "bf16", seed=14)
    pad = 4096
    n_o, n_l = B * H * S * d, B * H * S
    o_buf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    l_buf = torch.full((n_l + 2 * pad,), 7.0, dtype=torch.float32, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o = o_buf[pad:pad + n_o]
    lse = l_buf[pad:pad + n_l]
    attn_fwd(qd, kd, vd, o, lse, B, H, S, S, d, 1, 1 / math.sqrt(d), ATTN_DTYPE_BF16)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[pad + n_o:] == 7.0)
    assert torch.all(l_buf[:pad] == 7.0) and torch.all(l_buf[pad + n_l:] == 7.0)
    ro, rl = oracle.attention_forward(q, k, v, causal=True, scale=1 / math.sqrt(d))
    assert_parity(o.view(B, H, S, d), lse.view(B, H, S), ro, rl, "bf16", "canary")


def test_side_stream():
    q, k, v = make_qkv(2, 2, 400, 400, 64, "bf16", seed=15)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    ref_o, ref_l = fwd(qd, kd, vd, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fwd(qd, kd, vd, causal=True)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_host_buffers_entry_point():
    B, H, S, d = 1, 2, 500, 128
    q, k, v = make_qkv(B, H, S, S, d, "f16", seed=16)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    qd, kd, vd = torch.empty_like(q, device=DEV), torch.empty_like(k, device=DEV), torch.empty_like(v, device=DEV)
    od = torch.empty_like(q, device=DEV)
    ld = torch.empty((B, H, S), dtype=torch.float32, device=DEV)
    attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, B, H, S, S, d, 0, 1 / math.sqrt(d),
                  ATTN_DTYPE_F16)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=1 / math.sqrt(d))
    assert_parity(oh, lh, ro, rl, "f16", "host entry point")
    o2, l2 = fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=False)
    assert torch.equal(o2.cpu(), oh) and torch.equal(l2.cpu(), lh)


@pytest.mark.parametrize("B,H,S", [(2, 16, 2048), (1, 12, 4096), (1, 5, 8192)],
                         ids=["32-heads-weighted", "12-heads-equal", "5-heads-one-each"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_host_entry_point_pipelined_chunks(causal, B, H, S):
    """Above 32 MB the host entry point overlaps chunks of heads (8 chunks weighted
    1:3:...:3:1 from 20 heads on, 8 equal ones below that, one per head below 8);
    results match the device path."""
    d = 128
    q, k, v = make_qkv(B, H, S, S, d, "bf16", seed=18)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.full_like(qh, 3.0).pin_memory()
    lh = torch.full((B, H, S), 3.0, dtype=torch.float32).pin_memory()
    dev = [torch.empty_like(t, device=DEV) for t in (q, k, v, q)]
    ld = torch.empty((B, H, S), dtype=torch.float32, device=DEV)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        attn_fwd_host(qh, kh, vh, oh, lh, *dev, ld, B, H, S, S, d, int(causal), 1 / math.sqrt(d),
                      ATTN_DTYPE_BF16)
    side.synchronize()
    o2, l2 = fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o2.cpu(), oh) and torch.equal(l2.cpu(), lh)


def test_invalid_arguments_raise_on_gpu():
    q, k, v = make_qkv(1, 1, 64, 64, 96, "bf16", seed=17)
    with pytest.raises(AttnError) as e:
        fwd(q.to(DEV), k.to(DEV), v.to(DEV))
    assert "head_dim" in str(e.value)


def test_device_status_clean():
    attn_get_device_status()


def test_concurrent_host_threads_on_separate_streams():
    """Calls from two host threads on two streams give the single-threaded results."""
    import threading
    cases = [make_qkv(2, 4, 700, 700, 128, "bf16", seed=19 + i) for i in range(2)]
    dev = [tuple(t.to(DEV) for t in c) for c in cases]
    ref = [fwd(*qkv, causal=bool(i)) for i, qkv in enumerate(dev)]
    torch.cuda.synchronize()
    out = [None, None]
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                res = [fwd(*dev[i], causal=bool(i)) for _ in range(20)]
            s.synchronize()
            out[i] = res[-1]
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        assert torch.equal(out[i][0], ref[i][0]) and torch.equal(out[i][1], ref[i][1])
