"""The several-GPU form of the benchmark is replicas: every rank runs the
whole step on its own batch, and the job's time is the slowest rank's.  Its
host logic runs here as two gloo processes on the CPU."""
import os
import socket
import types

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(times[rank])
        q.put((rank, m, bench.job_rate(1000.0, world, m)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_the_whole_job_rate():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [2.5, 4.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, m, rate in got:
        assert m == 4.0  # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 1000.0 / 4.0e-3)  # units of both ranks over that time


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    def no_work(*a, **k):
        raise AssertionError("a rank other than 0 built the workload")

    monkeypatch.setattr(bench.wl, "make_config", no_work)
    args = types.SimpleNamespace(workload="shared_system_prompt", steps=1, warmup=3)
    assert bench.run_reference(args) == 0
