"""The N>1 host path on CPU: two gloo ranks.

Each rank runs its own replica of the work (weak scaling: no data-path
collective), the job time is the maximum over ranks, and the reported value
counts the work of every rank.  The per-rank compute here is the CPU oracle on
a small seeded workload, standing in for the GPU launch, whose data path is
the same on every rank.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from exact_attention_53_gb300.workloads import make_qkv

        # every rank: its own replica (same shapes, its own seed)
        q, k, v = make_qkv(1, 2, 64, 64, 16, "bf16", seed=100 + rank)
        o, lse = oracle.attention_forward(q, k, v, causal=True, scale=0.25)
        np.save(os.path.join(out_dir, f"o{rank}.npy"), o)
        # fake per-rank timings: the job time is the slowest rank's
        my_ms = 10.0 + 5.0 * rank
        job_ms = bench.max_over_ranks(my_ms, world)
        flops = 4.0 * 2 * 64 * 64 * 16 / 2
        value = bench.replica_throughput(flops, 3, world, job_ms)
        np.save(os.path.join(out_dir, f"t{rank}.npy"), np.array([job_ms, value]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_max_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    import oracle
    from exact_attention_53_gb300.workloads import make_qkv
    for rank in range(world):
        q, k, v = make_qkv(1, 2, 64, 64, 16, "bf16", seed=100 + rank)
        o_ref, _ = oracle.attention_forward(q, k, v, causal=True, scale=0.25)
        np.testing.assert_array_equal(np.load(tmp_path / f"o{rank}.npy"), o_ref)
        job_ms, value = np.load(tmp_path / f"t{rank}.npy")
        assert job_ms == 15.0                      # max over ranks, seen by every rank
        assert value == pytest.approx(4.0 * 2 * 64 * 64 * 16 / 2 * 3 * world / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_throughput(1e12, 10, 1, 1000.0) == pytest.approx(10.0)


def test_measured_traffic_is_tied_to_kernel_sources(tmp_path, monkeypatch):
    """The committed traffic record parses, and a figure counts only for unchanged sources."""
    import json
    import sys
    sys.path.insert(0, ROOT)
    import bench
    for key in bench.KERNEL_SOURCES:
        v = bench.measured_traffic(key)
        assert v is None or (isinstance(v, int) and v > 0)
    key = "attn_fwd_d128_bf16_full_c3"
    good = bench.kernel_source_digest(bench.KERNEL_SOURCES[key])
    (tmp_path / "profiles").mkdir()
    rec = {key: {"bytes": 123, "sources_sha256": good},
           "attn_fwd_d128_bf16_causal_c3": {"bytes": 456, "sources_sha256": "0" * 64},
           "attn_bwd_d128_bf16_full_c3": 789}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda names: good)
    assert bench.measured_traffic(key) == 123
    monkeypatch.setattr(bench, "kernel_source_digest", lambda names: "f" * 64)
    assert bench.measured_traffic(key) is None
    assert bench.measured_traffic("attn_bwd_d128_bf16_full_c3") is None
