#!/usr/bin/env python
"""Throughput of the chunked KDA forward on GB300 (one JSON line on stdout).

A step is one `kda_chunk_fwd` call (every launch of the hot path: offsets
pre-pass when packed, chunk prep, chunk scan) over the training-shape workload
B=1, T=8192, H=HV=16, K=V=128, bf16 q/k/v/beta, fp32 log2 gate, no initial
state, final state stored.  Inputs are synthetic (kda_synth) and resident in
HBM before the timed region; a 512 MiB buffer is written between timed steps
to flush the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the fp64 CPU oracle instead, on the host cores, each
step a bounded sample of the same workload.  Under torchrun (N > 1) every rank
runs its own replica of the workload (weak scaling, no collective on the data
path); rank 0 prints the line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunk_kda fwd tokens/s (T=8192,HV=16,K=V=128,bf16) and % of roofline on 1 GB300"
UNIT = "tokens/s"
WORKLOAD = 1
FLUSH_BYTES = 512 << 20


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ------------------------------------------------------------------ ranks
def max_over_ranks(x, dist=None, device="cpu"):
    """The largest of each rank's x (the job is as slow as its slowest rank)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, tokens_per_rank, ms):
    """Whole-job tokens/s: every rank processes its own replica of the workload
    (weak scaling), all in `ms` milliseconds (the max over ranks)."""
    return world * tokens_per_rank / (ms / 1e3)


# ------------------------------------------------------------------ bytes
def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def algorithmic_bytes(inp, ht_stored=True):
    """Compulsory HBM traffic of one forward: every input read once, o and the
    final state written once (no intermediate traffic counted)."""
    reads = sum(_nbytes(inp[n]) for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    w = inp["workload"]
    writes = _nbytes(inp["v"])  # o has v's shape and q's dtype (same dtype here)
    if ht_stored:
        writes += inp["N"] * w.HV * w.K * w.V * 4
    return reads, writes


def kernel_algorithmic_bytes(name, inp):
    """Compulsory bytes attributed to one kernel of the path."""
    r, wr = algorithmic_bytes(inp)
    state_in = _nbytes(inp["h0"])
    if name.startswith("chunk_prep"):
        return r - state_in
    if name.startswith("chunk_scan"):
        return wr + state_in
    if name.startswith("chunk_fused"):
        return r + wr
    return 0


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, interval_ms: int = 20):
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    f"-lms", str(interval_ms)]
        if gpu_id:
            self.cmd += ["-i", gpu_id]
        self.lines, self.proc, self.error = [], None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                         text=True)
        except OSError as e:
            self.error = str(e)
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"unsampled: {self.error}"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in timed region"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons)}


def _gpu_id(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:  # noqa: BLE001
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


def _traffic(kernel):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    if digest != rec.get("source_sha256_16"):
        return None
    return rec["dram_bytes_per_launch"]


# ------------------------------------------------------------------ CPU oracle
def cpu_oracle_rate(inp_cpu, budget_s=12.0, max_tokens=None):
    """Oracle tokens/s on the first L tokens (all heads) of the workload."""
    import oracle

    q, k, v, g, beta = (inp_cpu[n] for n in ("q", "k", "v", "g", "beta"))
    T = q.shape[1]
    L = min(T, max_tokens or T)
    sl = lambda t: t[:, :L]
    oracle.recurrent(sl(q)[:, :16], sl(k)[:, :16], sl(v)[:, :16], sl(g)[:, :16],
                     sl(beta)[:, :16], want_state=False)  # warm (loads the library)
    runs, t_total, toks = 0, 0.0, 0
    while t_total < budget_s or runs == 0:
        t0 = time.perf_counter()
        oracle.recurrent(sl(q), sl(k), sl(v), sl(g), sl(beta), h0=inp_cpu["h0"])
        t_total += time.perf_counter() - t0
        toks += L * q.shape[0]
        runs += 1
        if runs >= 3:
            break
    return toks / t_total, runs, L, oracle.num_threads()


def run_reference(args):
    """The oracle as the reference arm: each step one bounded sample."""
    import torch  # noqa: F401

    import kda_synth

    rank = _env_int("RANK", 0)
    if rank != 0:
        return 0
    inp = kda_synth.make_inputs(WORKLOAD, device="cpu")
    # Size a step so that warm-up + steps end within ~2 minutes.
    probe_rate, _, _, cores = cpu_oracle_rate(inp, budget_s=0.0, max_tokens=256)
    per_step_s = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    L = int(max(16, min(inp["q"].shape[1], probe_rate * per_step_s)))
    import oracle

    sl = lambda t: t[:, :L]
    for _ in range(args.warmup):
        oracle.recurrent(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g"]), sl(inp["beta"]))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrent(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g"]), sl(inp["beta"]))
    dt = time.perf_counter() - t0
    ms = 1e3 * dt / max(1, args.steps)
    value = L / (ms / 1e3)
    w = inp["workload"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.HV, "K": w.K,
                   "V": w.V, "input_dtype": "bf16", "sample_tokens_per_step": L},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {L} of {w.T} tokens, all {w.HV} heads, per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ ours
def run_ours(args):
    import torch

    import gated_delta_rule_cumsum_gb300 as kda
    import kda_synth

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    from gated_delta_rule_cumsum_gb300 import build as kbuild

    if rank == 0 or world == 1:
        kbuild.build()
    if dist:
        dist.barrier()
    kda.load()

    inp = kda_synth.make_inputs(WORKLOAD, device=dev)
    w = inp["workload"]
    q, k, v, g, beta, h0, cu = (inp[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    shape = kda.make_shape(q, v, cu)
    o = torch.empty_like(v)
    ht = torch.empty(inp["N"], w.HV, w.K, w.V, dtype=torch.float32, device=dev)
    ws = torch.empty(kda.kda_chunk_workspace_size(shape), dtype=torch.uint8, device=dev)
    status = kda.new_status(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.kda_chunk_fwd(q, k, v, g, beta, h0, cu, shape, o, ht, ws, status, stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    st, bits = kda.kda_read_device_status(status, stream)
    if st != 0:
        raise SystemExit(f"device status {bits:#x} after warm-up")

    sampler = ClockSampler(_gpu_id(torch, local)) if rank == 0 else None
    if sampler:
        sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.fill_(1.0)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    clocks = sampler.stop(t_wall0, t_wall1) if sampler else None
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps, dist,
                        dev)
    tokens = inp["tokens"]
    value = job_throughput(world, tokens, ms)

    # Per-kernel durations, live, with CUDA events on the launching stream.
    prof_steps = min(args.steps, 50)
    kda.kda_profile_reset()
    kda.kda_profile_enable(True)
    for _ in range(prof_steps):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    kda.kda_profile_enable(False)
    per_kernel = kda.kda_profile_report()
    kda.kda_profile_reset()
    launches_per_step = sum(c for _, c in per_kernel.values()) / prof_steps
    dom = max(per_kernel, key=lambda n: per_kernel[n][0])
    dom_ms = per_kernel[dom][0] / per_kernel[dom][1]
    peaks = _peaks()
    dom_bytes = kernel_algorithmic_bytes(dom, inp)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    traffic = _traffic(dom)
    r_b, w_b = algorithmic_bytes(inp)
    path_gbs = (r_b + w_b) / (ms / 1e3) / 1e9

    # End to end through the C ABI with host buffers: every step copies its inputs
    # from pinned host memory, runs the call and reads o and the final state back.
    # Pipelined: step i's H2D (copy stream) overlaps step i-1's call (compute
    # stream) and step i-2's D2H (copy-back stream), with two sets of device
    # inputs and outputs; events order each buffer's reuse.  The one-stream
    # sequential time is reported beside it.
    names = ("q", "k", "v", "g", "beta")
    host = {n: inp[n].cpu().pin_memory() for n in names}
    dev_in = [{n: torch.empty_like(inp[n]) for n in names} for _ in range(2)]
    dev_o = [torch.empty_like(o) for _ in range(2)]
    dev_ht = [torch.empty_like(ht) for _ in range(2)]
    o_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    ht_h = [torch.empty(ht.shape, dtype=ht.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(_nbytes(t) for t in host.values())
    d2h = _nbytes(o_h[0]) + _nbytes(ht_h[0])
    e2e_steps = min(args.steps, 30)
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_comp = torch.cuda.Stream(dev)

    def run_pipeline(nsteps):
        up_done = [torch.cuda.Event() for _ in range(nsteps)]
        comp_done = [torch.cuda.Event() for _ in range(nsteps)]
        down_done = [torch.cuda.Event() for _ in range(nsteps)]
        for i in range(nsteps):
            j = i % 2
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(comp_done[i - 2])  # buffer j's previous call has read it
                for n in names:
                    dev_in[j][n].copy_(host[n], non_blocking=True)
                up_done[i].record(s_up)
            s_comp.wait_event(up_done[i])
            if i >= 2:
                s_comp.wait_event(down_done[i - 2])  # outputs j have been read back
            d = dev_in[j]
            kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0, cu, shape, dev_o[j],
                              dev_ht[j], ws, status, s_comp)
            comp_done[i].record(s_comp)
            with torch.cuda.stream(s_down):
                s_down.wait_event(comp_done[i])
                o_h[j].copy_(dev_o[j], non_blocking=True)
                ht_h[j].copy_(dev_ht[j], non_blocking=True)
                down_done[i].record(s_down)
        return down_done[nsteps - 1]

    run_pipeline(3)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    last = run_pipeline(e2e_steps)
    last.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / e2e_steps, dist, dev)
    e2e_value = job_throughput(world, tokens, e2e_ms)

    def seq_step():
        d = dev_in[0]
        for n in names:
            d[n].copy_(host[n], non_blocking=True)
        kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0, cu, shape, dev_o[0],
                          dev_ht[0], ws, status, stream)
        o_h[0].copy_(dev_o[0], non_blocking=True)
        ht_h[0].copy_(dev_ht[0], non_blocking=True)

    for _ in range(3):
        seq_step()
    torch.cuda.synchronize(dev)
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_s.record(stream)
    for _ in range(e2e_steps):
        seq_step()
    e_e.record(stream)
    torch.cuda.synchronize(dev)
    e2e_seq_ms = max_over_ranks(e_s.elapsed_time(e_e) / e2e_steps, dist, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_cpu = {n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in inp.items()}
        rate, runs, L, cores = cpu_oracle_rate(inp_cpu, budget_s=10.0)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"full workload ({L} tokens x {w.HV} heads), {runs} run(s), fp64"}

    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    # bf16 operands with fp32 accumulation on the tensor-core path; fp32 on the SIMT path
    compute_dtype = "bf16" if any(n.endswith("_tc") for n in per_kernel) else "f32"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": compute_dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.HV, "K": w.K,
                   "V": w.V, "input_dtype": "bf16", "gate_dtype": "f32", "h0": "none",
                   "ht": "stored", "l2_flush": "512 MiB write between timed steps",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": traffic, "algorithmic_bytes": dom_bytes,
                     "kernel_ms": dom_ms, "peak_source": peaks["source"],
                     "path_gbs": path_gbs, "path_frac": path_gbs / peaks["hbm_gbs"]},
        "kernels": {n: {"ms_per_launch": t / c, "launches_per_step": c / prof_steps}
                    for n, (t, c) in per_kernel.items()},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "mode": "pipelined: step i's H2D overlaps step i-1's call and step i-2's D2H "
                        "(two buffer sets, three streams; wall clock over the steps)",
                "sequential_ms_per_step": e2e_seq_ms},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
