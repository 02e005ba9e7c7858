"""The N > 1 host logic of bench.py on CPU: world-size-2 `gloo` ranks run the
bench's own barrier, max-over-ranks and whole-job aggregation, and the
reference arm's rank rule.  The path has no data-path collective (replicas
only), so these host steps are all that N > 1 adds."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench._barrier(world, torch)
        # rank r took (r + 1) * 10 ms for 5 steps of 1e9 bytes each
        ms_step, gbs = bench._job_rate(10.0 * (rank + 1), 5, 1e9, world, torch, "cpu")
        bench._barrier(world, torch)
        out[rank] = (ms_step, gbs)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_with_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    # both ranks see the slowest rank's time (20 ms / 5 steps = 4 ms per step)
    # and the aggregate counts both ranks' bytes: 2 * 1e9 B / 4 ms = 500 GB/s
    for r in range(world):
        ms_step, gbs = out[r]
        assert ms_step == pytest.approx(4.0)
        assert gbs == pytest.approx(500.0)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench._max_over_ranks(3.5, 1, torch, "cpu") == 3.5
    ms_step, gbs = bench._job_rate(8.0, 4, 2e9, 1, torch, "cpu")
    assert ms_step == pytest.approx(2.0) and gbs == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_0_only():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup = 1, 3
    assert bench.run_reference(A(), 1, 2) is None     # other ranks exit without work


def test_reference_arm_line_on_rank_0():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup = 1, 0
    res = bench.run_reference(A(), 0, 1)
    assert res["impl"] == "reference" and res["unit"] == "GB/s" and res["value"] > 0
    assert res["cpu_baseline"]["value"] == res["value"] and res["cpu_baseline"]["kind"] == "oracle"
    assert res["e2e"] == {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
