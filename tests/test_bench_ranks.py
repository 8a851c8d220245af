"""The benchmark's multi-process path on CPU: world size 2 over gloo (127.0.0.1).

One process per GPU, no collective on the data path: the only cross-rank step is the timing
reduction (the job takes as long as its slowest rank) and the whole-job throughput (every rank
processes its own lanes: weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        out.put((rank, ms, bench.job_throughput(world, 8 * 40960, ms)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_the_whole_job():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    times = [1.25, 1.75]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for rank, ms, value in res:
        assert ms == 1.75                                   # the slower rank's time, on every rank
        assert value == pytest.approx(2 * 8 * 40960 / 1.75e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.job_throughput(1, 1000, 2.0) == pytest.approx(5.0e5)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun only rank 0 times the oracle; the other ranks exit 0 without work."""
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(argparse.Namespace(steps=1, warmup=0, seed=0)) == 0
