"""The benchmark's multi-rank host logic on CPU: two gloo ranks, as under torchrun.

Each rank of `bench.py --gpus N` runs an independent replica of the workload (no data-path
collective); the job's time is the slowest rank's and its throughput counts every rank's bytes.
The reference arm runs on rank 0 only; other ranks leave without work.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        elapsed = 10.0 + 5.0 * rank  # rank 1 is the slow one
        mx = bench.max_over_ranks(elapsed, dist, "cpu")
        dist.barrier()
        q.put((r, ws, local, mx, bench.job_gbs(1e9, ws, mx)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for r, (rank, ws, local, mx, gbs) in enumerate(res):
        assert (rank, ws, local) == (r, 2, r)
        assert mx == 15.0  # both ranks see the slowest rank's time
        assert gbs == pytest.approx(2e9 / 15e-3 / 1e9)  # 2 ranks x 1 GB over 15 ms


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_gbs(2e9, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 3, 1

    assert bench.run_reference(A()) is None
    assert capsys.readouterr().out == ""
