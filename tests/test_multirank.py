"""bench.py's multi-rank host logic on CPU: two gloo ranks (one process each).

Each GPU runs its own full copy of the workload (replicas; the operator needs no
exchange), so the only cross-rank steps are a barrier and the max of the per-rank step
times; the job's value is world x work / that max.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        step_ms = 2.0 + rank                      # rank 1 is the slow one
        out[rank] = bench.max_over_ranks(step_ms, world)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == 3.0


def test_whole_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tflops(1, 2.0e12, 1.0)
    assert one == pytest.approx(2000.0)
    assert bench.whole_job_tflops(4, 2.0e12, 1.0) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
