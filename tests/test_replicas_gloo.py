"""Several GPUs run replicas only: the GEMM has no exchange step, so each rank runs its
own copy of the workload; the job is timed by the slowest rank and its throughput
counts every rank's work (weak scaling).  The host side of that path is checked here
with two gloo ranks on the CPU; the reference arm runs on rank 0 alone.
"""
import io
import os
import socket
import contextlib

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        local_ms = 10.0 + 5.0 * rank                    # rank 1 is the slower replica
        slowest = bench.max_over_ranks(local_ms, torch.device("cpu"))
        q.put((rank, ws, r, local, slowest, bench.replica_throughput(ws, 1e12, 4, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_are_timed_by_the_slowest_and_count_both_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for rank, (r0, ws, r, local, slowest, tflops) in enumerate(got):
        assert (r0, ws, r, local) == (rank, 2, rank, rank)
        assert slowest == 15.0
        # 2 replicas x 4 steps x 1 TFLOP in 15 ms
        assert tflops == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_without_a_process_group_the_local_time_is_the_job_time():
    import bench
    assert bench.max_over_ranks(7.5, torch.device("cpu")) == 7.5
    assert bench.replica_throughput(1, 2e12, 10, 20.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(None) == 0        # returns before touching its arguments
    assert out.getvalue() == ""
