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


def _layout(B, T, HV=2, K=8, V=8, cu=None, h0=True, N=None):
    import torch

    q = torch.zeros(B, T, 1, K)
    N = N if N is not None else (B if cu is None else len(cu) - 1)
    return dict(q=q, k=q.clone(), v=torch.zeros(B, T, HV, V), g=torch.zeros(B, T, HV, K),
                beta=torch.zeros(B, T, HV), h0=torch.zeros(N, HV, K, V) if h0 else None,
                cu_seqlens=None if cu is None else torch.tensor(cu, dtype=torch.int32))


def test_oracle_sample_packed_takes_whole_sequences_and_skips_leading_empty_slots():
    inp = _layout(1, 100, cu=[0, 0, 30, 30, 70, 90])
    part, L, _ = bench.oracle_sample(inp, 5)  # smaller than the first sequence
    assert L == 30 and part["cu_seqlens"].tolist() == [0, 0, 30]
    assert part["q"].shape[1] == 30 and part["h0"].shape[0] == 2
    part, L, _ = bench.oracle_sample(inp, 75)
    assert L == 70 and part["cu_seqlens"].tolist() == [0, 0, 30, 30, 70]
    assert part["h0"].shape[0] == 4
    part, L, _ = bench.oracle_sample(inp, 10 ** 6)
    assert L == 90 and part["cu_seqlens"].tolist() == [0, 0, 30, 30, 70, 90]


def test_oracle_sample_dense_batches_and_long_sequences():
    inp = _layout(4096, 1)  # decode: one token per sequence
    part, L, _ = bench.oracle_sample(inp, 64)
    assert L == 64 and part["q"].shape[:2] == (64, 1) and part["h0"].shape[0] == 64
    inp = _layout(1, 8192, h0=False)  # one long sequence: a token prefix
    part, L, _ = bench.oracle_sample(inp, 1000)
    assert L == 1000 and part["q"].shape[:2] == (1, 1000) and part["h0"] is None
    inp = _layout(4, 256)
    part, L, _ = bench.oracle_sample(inp, 600)
    assert L == 512 and part["q"].shape[:2] == (2, 256)


def test_derived_fp32_peak_and_recurrence_flops():
    # 152 SMs x 128 lanes x 2 flops x 2070 MHz
    assert bench.fp32_fma_tflops(152, 2070.0) == pytest.approx(80.55, abs=0.01)

    class W:
        HV, K, V = 32, 128, 128

    assert bench.recurrent_flops({"tokens": 4096 * 256, "workload": W}) == \
        7 * 4096 * 256 * 32 * 128 * 128


def test_every_bench_workload_exists_in_the_generator():
    import kda_synth

    for name, (idx, over, steps, warm) in bench.WORKLOADS.items():
        w = kda_synth.workload(idx, **over)
        assert steps >= 1 and warm >= 3, name
        assert (name in bench.RECURRENT) == bool(w.decode_seqs), name


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` end to end on the host (the oracle timed on a bounded
    sample): one JSON line with the arm's keys, its e2e moving nothing."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["n_gpus"] == 1 and d["higher_is_better"] is True and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("train_bf16_B1_T8192")
    # the same config keys and values as the GPU arm's line (both come from the
    # workload's definition), so the two lines compare as one workload
    sys.path.insert(0, root)
    import bench

    assert d["config"] == bench.workload_config("train")
