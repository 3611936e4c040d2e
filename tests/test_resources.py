"""Build-time resource checks (CPU only; needs nvcc).

Every kernel instantiation is compiled with ``-Xptxas -v`` (the build's own flags) and must not
spill, and the two-tile forward kernels and the dK/dV and dQ backward kernels must launch with
exactly the 168 registers per thread that their warpgroup register splits assume (the host
refuses to launch them otherwise, so a drift here would only show up on a GPU).
"""

import re

import pytest


@pytest.fixture(scope="module")
def table():
    from exact_attention_53_gb300 import build as b
    try:
        b._nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    rows = {}
    for line in b.resources().splitlines()[2:]:
        cells = [c.strip() for c in line.strip("|").split("|")]
        rows[cells[0].strip("`")] = tuple(int(x) for x in cells[1:])
    return rows


def test_every_kernel_reported(table):
    from exact_attention_53_gb300.build import BWD_INSTANCES, INSTANCES
    fwd = [k for k in table if "attn_fwd_kernel" in k]
    bwd = [k for k in table if re.search(r"attn_bwd_(dkdv|dq|prep)_kernel", k)]
    wide = [k for k in table if "attn_bwd_wide_kernel" in k]
    assert len(fwd) == len(INSTANCES)
    # per instance: dQ, and dK/dV (d <= 128) or its two d = 256 passes; prep per (d, dtype)
    n_wide = sum(1 for d, _, _ in BWD_INSTANCES if d == 256)
    assert len(bwd) == 2 * len(BWD_INSTANCES) - n_wide + len(BWD_INSTANCES) // 2
    assert len(wide) == 2 * n_wide


def test_no_kernel_spills(table):
    spilling = {k: v for k, v in table.items() if v[3] or v[4]}
    assert not spilling, f"register spills: {spilling}"


def test_two_tile_forward_launch_registers(table):
    # (head dim, split): head dims 64 and 128 without split-KV run two query tiles per CTA
    for name, (regs, *_rest) in table.items():
        m = re.match(r"attn::attn_fwd_kernel<\(int\)(\d+), \(bool\)\d, \(bool\)\d, \(bool\)(\d)>", name)
        if m and int(m.group(1)) in (64, 128) and m.group(2) == "0":
            assert regs == 168, f"{name}: {regs} registers at launch, the split expects 168"


def test_backward_launch_registers(table):
    # the dK/dV and dQ kernels (d = 64, 128 and the d = 256 dQ) run 384 threads re-split from 168
    found = 0
    for name, (regs, *_rest) in table.items():
        if re.match(r"attn::attn_bwd_(dkdv|dq)_kernel<", name):
            found += 1
            assert regs == 168, f"{name}: {regs} registers at launch, the split expects 168"
    assert found > 0
