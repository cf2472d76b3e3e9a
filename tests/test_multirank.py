"""bench.py's multi-GPU host logic on CPU: two gloo ranks (weak scaling, one
replica of the workload per rank, job time = the slowest rank)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms_local = 1.5 + rank  # rank 1 is the slowest
        ms = bench.max_over_ranks(ms_local, dist, "cpu")
        value = bench.job_throughput(world, 8192, ms)
        dist.barrier()
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == 2.5  # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 8192 / 2.5e-3)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.job_throughput(1, 1000, 2.0) == pytest.approx(5e5)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 5, 3, 2

    assert bench.run_reference(A()) == 0
