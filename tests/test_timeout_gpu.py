"""GPU failure detection: a wait that runs out, or a launch past its deadline, is
reported and does not hang.

The debug build of the forward kernel (libattn_debug.so, include/attn_debug.h)
waits at most 1 ms per barrier, can be told to load nothing for one work unit,
and takes its CTAs' time budget as an argument.  Nothing faults or hangs: a
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
from exact_attention_53_gb300 import attn_get_device_status, fwd
from exact_attention_53_gb300.binding import load_debug_library
from exact_attention_53_gb300.workloads import make_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
# status bits of the debug library's roles (include/attn_debug.h)
PRODUCER, MMA, SOFTMAX, EPILOGUE, DRAIN, DEADLINE = 1, 2, 4, 8, 16, 512


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
