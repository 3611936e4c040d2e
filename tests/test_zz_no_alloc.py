"""GPU test of the allocation-free split-KV entry point (attn_fwd_splitkv_noalloc).

It must give exactly the results of the workspace entry point
(attn_fwd_splitkv) on the same inputs -- the same kernels over the same key
ranges, so bit for bit -- call after call, although every call reuses the one
built-in scratch array.  The file is named to be collected last, so that in a
full run it also executes after every other GPU test has used the library.
"""

import math

import pytest
import torch

import oracle
from exact_attention_53_gb300 import (AttnError, attn_fwd_splitkv_noalloc, attn_fwd_splitkv_plan,
                                      attn_get_device_status, fwd_splitkv)
from exact_attention_53_gb300.binding import NOALLOC_SCRATCH_BYTES
from exact_attention_53_gb300.workloads import make_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")
DTYPE_CODE = {"f16": 0, "bf16": 1}
BF16_TOL = 1e-2        # |ΔO| bound of the bf16 parity tolerance at |O| ≲ 1 (absolute part)
F16_TOL = 4e-3
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_53_gb300.build import build
    build()
    yield
    attn_get_device_status()


def _noalloc(q, k, v, n_split, scale, dtype):
    B, H, S_q, d = q.shape
    S_k = k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
    attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, S_q, S_k, d, scale, DTYPE_CODE[dtype],
                             n_split)
    return o, lse


CASES = [  # (B, H, S_q, S_k, d, dtype, n_split)
    (2, 16, 1, 32768, 128, "bf16", 0),
    (1, 4, 37, 9000, 64, "f16", 7),
    (1, 2, 130, 5000, 256, "bf16", 3),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + f"-{c[5]}-n{c[6]}")
def test_two_calls_in_a_row_match_the_workspace_entry_point(case):
    B, H, S_q, S_k, d, dtype, n_split = case
    n, ws = attn_fwd_splitkv_plan(B, H, S_q, S_k, d, DTYPE_CODE[dtype], n_split)
    assert n > 1 and 0 < ws <= NOALLOC_SCRATCH_BYTES
    scale = 1 / math.sqrt(d)
    tol = BF16_TOL if dtype == "bf16" else F16_TOL
    # Two different inputs back to back on one stream: the second call reuses
    # the scratch the first one wrote.
    inputs = [make_qkv(B, H, S_q, S_k, d, dtype, seed=900 + i) for i in range(2)]
    dev_inputs = [tuple(t.to(DEV) for t in qkv) for qkv in inputs]
    outs = [_noalloc(*qkv, n_split, scale, dtype) for qkv in dev_inputs]
    refs = [fwd_splitkv(*qkv, n_split=n_split, scale=scale) for qkv in dev_inputs]
    torch.cuda.synchronize()
    for (o, lse), (ro, rl) in zip(outs, refs):
        assert (o.float() - ro.float()).abs().max().item() <= tol
        assert (lse - rl).abs().max().item() <= LSE_TOL
        assert torch.equal(o, ro) and torch.equal(lse, rl)
    # and the second call against the oracle
    q, k, v = inputs[1]
    eo, el = oracle.attention_forward(q, k, v, causal=False, scale=scale)
    assert_parity(outs[1][0], outs[1][1], eo, el, dtype, "noalloc second call")


def test_one_range_needs_no_scratch():
    q, k, v = (t.to(DEV) for t in make_qkv(1, 2, 20, 100, 64, "bf16", seed=910))
    o, lse = _noalloc(q, k, v, 0, 0.125, "bf16")
    ro, rl = fwd_splitkv(q, k, v, n_split=0, scale=0.125)
    torch.cuda.synchronize()
    assert torch.equal(o, ro) and torch.equal(lse, rl)


def test_plan_above_the_scratch_is_rejected_on_a_gpu():
    B, H, S_q, S_k, d = 4, 32, 256, 16384, 128
    q, k, v = (torch.empty((B, H, S, d), dtype=torch.bfloat16, device=DEV)
               for S in (S_q, S_k, S_k))
    with pytest.raises(AttnError, match="scratch"):
        _noalloc(q, k, v, 64, 0.125, "bf16")
