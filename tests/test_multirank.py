"""The benchmark's multi-rank aggregation on CPU: two gloo ranks with different
timings must both report the job throughput of two replicas over the slower
rank's time (the path shards by sequence with no exchange, so ranks are
independent replicas and only the timing is reduced)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import sys

    import torch.distributed as dist

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total_ms = [30.0, 45.0][rank]  # rank 1 is the slower one
        ms_step, per_s = bench.job_throughput(total_ms, steps=10, units_per_step=1e6,
                                              world=world, device="cpu")
        results[rank] = (ms_step, per_s)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        ms_step, per_s = results[r]
        assert ms_step == pytest.approx(4.5)                # 45 ms / 10 steps
        assert per_s == pytest.approx(2 * 1e6 / 4.5e-3)    # both replicas' units


def test_single_rank_needs_no_process_group():
    import bench

    ms_step, per_s = bench.job_throughput(20.0, steps=4, units_per_step=100.0, world=1)
    assert ms_step == 5.0 and per_s == pytest.approx(100.0 / 5e-3)
