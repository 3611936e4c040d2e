"""GPU failure detection: a wait that runs out, or a launch past its deadline, is
reported and does not hang.

The debug build of the forward and backward kernels (libattn_debug.so,
include/attn_debug.h) waits at most 1 ms per barrier, can be told to load
nothing for one work unit (the forward's, or the backward dK/dV kernel's), and
takes its CTAs' time budget as an argument.  Nothing faults or hangs: a
skipped unit's consumers wait on barriers nothing completes and their waits run
out; a launch given a budget shorter than its work has its producers stop
their CTAs at the deadline.  Either way the kernel records it in its status
word, stops the launch's other CTAs, frees tensor memory and returns.  These
tests check that the status reports it, that the call returns in
milliseconds, and that the same device then still computes correct results
with both the debug and the release library.
"""

import ctypes
import math
import time

import numpy as np
import pytest
import torch

import oracle
from exact_attention_53_gb300 import attn_get_device_status, bwd, fwd
from exact_attention_53_gb300.binding import load_debug_library
from exact_attention_53_gb300.workloads import make_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
# status bits of the debug library's roles (include/attn_debug.h)
PRODUCER, MMA, SOFTMAX, EPILOGUE, DRAIN, DEADLINE = 1, 2, 4, 8, 16, 512
BWD_PRODUCER, BWD_MMA, BWD_SOFTMAX, BWD_DRAIN, BWD_EPILOGUE = 32, 64, 128, 256, 1024


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_53_gb300.build import build
    build()
    yield
    attn_get_device_status()


def _run_debug(q, k, v, skip_unit, budget_ns=0):
    lib = load_debug_library()
    B, H, S, _ = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.monotonic()
    rc = lib.attn_debug_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, S, 1 / math.sqrt(64), skip_unit, budget_ns,
                            stream)
    assert rc == 0, f"launch returned cudaError {rc}"
    status = ctypes.c_uint(0)
    rc = lib.attn_debug_status(ctypes.byref(status), stream)
    elapsed = time.monotonic() - t0
    assert rc == 0, f"status read returned cudaError {rc}"
    return o, lse, status.value, elapsed


def _inputs(B, H, S, seed):
    q, k, v = make_qkv(B, H, S, S, 64, "bf16", seed=seed)
    return (q, k, v), tuple(t.to(DEV) for t in (q, k, v))


def _check_usable(host, dev_in, what):
    """The debug kernel without a skipped unit, then the release library, both match the oracle."""
    q, k, v = host
    ro, rl = oracle.attention_forward(q, k, v, causal=False, scale=1 / math.sqrt(64))
    o, lse, status, _ = _run_debug(*dev_in, skip_unit=-1)
    assert status == 0, f"{what}: a clean debug run reported status {status:#x}"
    assert_parity(o, lse, ro, rl, "bf16", f"{what}: debug library, no unit skipped")
    o2, l2 = fwd(*dev_in, causal=False)
    torch.cuda.synchronize()
    attn_get_device_status()
    assert_parity(o2, l2, ro, rl, "bf16", f"{what}: release library after the timeout")


def test_single_unit_wait_runs_out_and_is_reported():
    host, dev_in = _inputs(1, 1, 128, seed=71)
    o, lse, status, elapsed = _run_debug(*dev_in, skip_unit=0)
    # The MMA warp waits for a Q tile that never comes; the softmax and store
    # warps wait for work that never comes.  Any of them may run out first.
    assert status != 0, "no wait ran out although the unit's loads were skipped"
    assert status & ~(MMA | SOFTMAX | EPILOGUE) == 0, f"unexpected status bits {status:#x}"
    assert elapsed < 2.0, f"the call took {elapsed:.3f} s with 1 ms waits"
    _check_usable(host, dev_in, "single unit")


def test_one_unit_of_a_large_grid_stops_only_that_launch():
    # 2 x 64 heads x 2 query blocks = 256 work units over the work queue; unit 77 is skipped.
    host, dev_in = _inputs(2, 64, 512, seed=72)
    o, lse, status, elapsed = _run_debug(*dev_in, skip_unit=77)
    assert status != 0 and status & ~(MMA | SOFTMAX | EPILOGUE) == 0, f"status {status:#x}"
    assert elapsed < 2.0, f"the call took {elapsed:.3f} s with 1 ms waits"
    # The skipped unit (head 38, query rows 256..511) was never written.
    o_cpu = o.float().cpu().numpy()
    assert np.isnan(o_cpu[0, 38, 256:]).all()
    _check_usable(host, dev_in, "grid of 256 units")


def test_launch_past_its_deadline_stops_and_is_reported():
    # 4 x 64 heads x 8 query blocks = 2048 units of 16 key tiles (about 0.5 ms of work); each
    # CTA gets 30 µs, so the producers stop their CTAs and the rest of the launch stops too.
    host, dev_in = _inputs(4, 64, 2048, seed=74)
    o, lse, status, elapsed = _run_debug(*dev_in, skip_unit=-1, budget_ns=30_000)
    assert status & DEADLINE, f"status {status:#x} lacks the deadline bit"
    assert elapsed < 2.0, f"the call took {elapsed:.3f} s"
    # Units that started late were never computed: the launch really stopped early.
    assert torch.isnan(lse).any()
    _check_usable(host, dev_in, "deadline")


def test_status_is_clear_after_being_read():
    _, dev_in = _inputs(1, 1, 128, seed=73)
    _, _, first, _ = _run_debug(*dev_in, skip_unit=0)
    assert first != 0
    lib = load_debug_library()
    status = ctypes.c_uint(123)
    assert lib.attn_debug_status(ctypes.byref(status), torch.cuda.current_stream().cuda_stream) == 0
    assert status.value == 0


def _run_debug_bwd(dev_in, o, lse, dout, skip_unit, budget_ns=0):
    """One debug-build backward; returns dq, dk, dv (NaN where never written), status, seconds."""
    lib = load_debug_library()
    q, k, v = dev_in
    B, H, S, _ = q.shape
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    s_pad = (S + 127) // 128 * 128
    ws = torch.empty(2 * B * H * s_pad, dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.monotonic()
    rc = lib.attn_debug_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                            ws.data_ptr(), B, H, S, 1 / math.sqrt(64), skip_unit, budget_ns, stream)
    assert rc == 0, f"launch returned cudaError {rc}"
    status = ctypes.c_uint(0)
    rc = lib.attn_debug_status(ctypes.byref(status), stream)
    elapsed = time.monotonic() - t0
    assert rc == 0, f"status read returned cudaError {rc}"
    return dq, dk, dv, status.value, elapsed


def _bwd_inputs(B, H, S, seed):
    _, dev_in = _inputs(B, H, S, seed)
    o, lse = fwd(*dev_in, causal=False)
    dout = make_qkv(B, H, S, 1, 64, "bf16", seed=seed + 1)[0].to(DEV)
    torch.cuda.synchronize()
    return dev_in, o, lse, dout


def _check_bwd_usable(dev_in, o, lse, dout, what):
    """A clean debug backward, and then the release one, give the same bits."""
    dq, dk, dv, status, _ = _run_debug_bwd(dev_in, o, lse, dout, skip_unit=-1)
    assert status == 0, f"{what}: a clean debug backward reported status {status:#x}"
    ref = bwd(*dev_in, o, lse, dout, causal=False)
    torch.cuda.synchronize()
    attn_get_device_status()
    for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        assert torch.equal(got, want), f"{what}: {name} of the debug build differs from the release"


def test_backward_wait_runs_out_and_is_reported():
    # 2 heads x 2 key tiles = 4 dK/dV units; unit 1 (head 0, keys 128..255) is skipped.
    dev_in, o, lse, dout = _bwd_inputs(1, 2, 256, seed=75)
    dq, dk, dv, status, elapsed = _run_debug_bwd(dev_in, o, lse, dout, skip_unit=1)
    # The dK/dV MMA warp waits for K/V that never come; the softmax and epilogue warps
    # wait for work that never comes.  Any of them may run out first.
    assert status != 0, "no wait ran out although the unit's loads were skipped"
    allowed = BWD_PRODUCER | BWD_MMA | BWD_SOFTMAX | BWD_DRAIN | BWD_EPILOGUE
    assert status & ~allowed == 0, f"unexpected status bits {status:#x}"
    assert elapsed < 2.0, f"the call took {elapsed:.3f} s with 1 ms waits"
    # The skipped unit's key rows were never written; the dQ kernel ran to the end.
    assert torch.isnan(dk[0, 0, 128:].float()).all() and torch.isnan(dv[0, 0, 128:].float()).all()
    assert not torch.isnan(dq.float()).any()
    _check_bwd_usable(dev_in, o, lse, dout, "backward unit skipped")


def test_backward_launch_past_its_deadline_stops_and_is_reported():
    # 2 x 32 heads x 16 key tiles = 1024 dK/dV units (roughly 0.1 ms of work each way);
    # each CTA gets 30 µs, so the producers stop their CTAs and the rest of the launch stops.
    dev_in, o, lse, dout = _bwd_inputs(2, 32, 2048, seed=76)
    dq, dk, dv, status, elapsed = _run_debug_bwd(dev_in, o, lse, dout, skip_unit=-1, budget_ns=30_000)
    assert status & DEADLINE, f"status {status:#x} lacks the deadline bit"
    assert elapsed < 2.0, f"the call took {elapsed:.3f} s"
    assert torch.isnan(dk.float()).any()
    _check_bwd_usable(dev_in, o, lse, dout, "backward deadline")
