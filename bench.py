#!/usr/bin/env python
"""Throughput of the chunked KDA forward on GB300 (one JSON line on stdout).

A step is one `kda_chunk_fwd` call (every launch of the hot path: offsets
pre-pass when packed, chunk prep, chunk scan) over the training-shape workload
B=1, T=8192, H=HV=16, K=V=128, bf16 q/k/v/beta, fp32 log2 gate, no initial
state, final state stored.  Inputs are synthetic (kda_synth) and resident in
HBM before the timed region; a 512 MiB buffer is written between timed steps
to flush the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload train|train_wide_gate|gva|packed|decode|decode_small|prefill|prefill_small|
                              train_bwd|train_bwd_recurrent|train_step]

`--workload` picks one of the other synthetic workloads instead (grouped value
heads B4 T4096 HV32; packed varlen H=HV=32; decode 4096 x 1 token; its
256-token prefill variant); decode and prefill steps are one in-place
`kda_recurrent_fwd` call, a train_bwd step is one `kda_chunk_bwd` call (the
gradients of the training shape for dL/do and dL/dht drawn once, in the chunked
form on the tensor cores) and a train_bwd_recurrent step one `kda_recurrent_bwd`
call (the same gradients by the token recurrence); a train_step step is the
forward that keeps the backward's state (`kda_chunk_fwd_save`: o and ht) followed
by the backward from it (`kda_chunk_bwd` with KDA_FLAG_BWD_SAVED), a training
step's work on this layer.  `--impl reference` times the fp64 CPU oracle
instead, on the host cores, each step a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling, no collective on the data path); rank 0 prints the line with the
max-over-ranks time.
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
FLUSH_BYTES = 512 << 20
# name -> (kda_synth workload, overrides, default steps, default warm-up)
WORKLOADS = {
    "train": (1, {}, 2000, 20),
    # the training shape with per-token gates of -U(1.5, 3) (log2): every chunk's gate
    # range (~144) past the split grams', so every chunk takes the exact-gram path
    "train_wide_gate": (1, {"g_lo": 1.5, "g_hi": 3.0}, 500, 10),
    "gva": (2, {}, 500, 10),
    "packed": (3, {}, 300, 10),
    "decode": (4, {}, 100, 5),
    "prefill": (4, {"T": 256}, 10, 3),
    # the prefill variant on 256 of the 4096 sequences: the size an ncu capture takes
    "prefill_small": (4, {"T": 256, "B": 256, "decode_seqs": 256}, 20, 3),
    # decode on 512 of the 4096 sequences (1 GiB of state): the size an ncu capture takes
    "decode_small": (4, {"B": 512, "decode_seqs": 512}, 100, 5),
    # gradients of the training shape: chunked on the tensor cores (kda_chunk_bwd) and
    # by the token recurrence (kda_recurrent_bwd)
    "train_bwd": (1, {}, 50, 5),
    "train_bwd_recurrent": (1, {}, 10, 3),
    # forward (keeping the backward's state) + backward from it, the training shape
    "train_step": (1, {}, 50, 5),
}
BACKWARD = ("train_bwd", "train_bwd_recurrent", "train_step")
CHUNK_BWD = ("train_bwd", "train_step")
BWD_FLOPS_PER_ELEMENT = 26   # one forward pass (7) + the reverse sweep (19) per state element
RECURRENT = ("decode", "decode_small", "prefill", "prefill_small")
FP32_LANES_PER_SM = 128      # fp32 FMA lanes per SM (4 partitions x 32)
E2E_MAX_H2D = 8 << 30        # larger inputs are not staged through pinned host memory


def _metric(name, w):
    if name == "train":
        return METRIC
    if name == "train_wide_gate":
        return f"chunk_kda fwd tokens/s ({w.name}, gates -U(1.5,3) log2 per token) on 1 GB300"
    if name == "train_bwd":
        return f"chunk_kda bwd tokens/s ({w.name}) on 1 GB300"
    if name == "train_step":
        return f"chunk_kda fwd+bwd tokens/s ({w.name}) on 1 GB300"
    if name == "train_bwd_recurrent":
        return f"recurrent_kda bwd tokens/s ({w.name}) on 1 GB300"
    op = "recurrent_kda" if name in RECURRENT else "chunk_kda"
    return f"{op} fwd tokens/s ({w.name}) on 1 GB300"


def _make_inputs(name, device):
    import kda_synth

    idx, over, _, _ = WORKLOADS[name]
    return kda_synth.make_inputs(kda_synth.workload(idx, **over), device=device)


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
                "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


def fp32_fma_tflops(sms, sm_mhz):
    """Plain fp32 FMA peak: SMs x 128 lanes x 2 flops per FMA x SM clock."""
    return sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


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
    if name.startswith("chunk_fused") or name.startswith("recurrent"):
        return r + wr
    return 0


def chunk_bwd_bytes(inp):
    """Compulsory HBM traffic of one chunked backward: q, k, v, g, beta, dL/do and
    dL/dht read once; dq, dk, dv, dg, dbeta (fp32) and dh0 written once."""
    w = inp["workload"]
    reads = sum(_nbytes(inp[n]) for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    reads += _nbytes(inp["v"]) + inp["N"] * w.HV * w.K * w.V * 4          # do, dht
    rows = inp["q"].shape[0] * inp["q"].shape[1]
    writes = 4 * rows * (2 * w.H * w.K + w.HV * (w.V + w.K + 1))           # dq dk dv dg dbeta
    writes += inp["N"] * w.HV * w.K * w.V * 4                              # dh0
    return reads, writes


def chunk_bwd_flops(inp):
    """Useful tensor-core flops of one chunked backward per (64-row chunk, value
    head), K = V = 128, counted from the products the seven stages form:
    recompute + re-scan (the forward's 1.41e5 per token-head x 64), the reverse
    state scan (Aqk^T do, kg dh, qg^T do, w^T dv': 7.3e6) and the per-chunk
    gradients (P, do v'^T, [do; dv'] h^T, v' dh^T, dAkk, Akk^T [dv' | dw],
    Akk^T dAkk, X Akk^T, [dP; dA] kn, dP^T kp + dA^T qp: 1.78e7)."""
    w = inp["workload"]
    units = inp["tokens"] / 64 * w.HV
    return units * (64 * 1.41e5 + 7.3e6 + 1.78e7)


def chunk_bwd_roofline(inp, per_kernel, prof_steps, ms, peaks, name, with_forward_outputs=False):
    """The whole call against the tighter of HBM (its compulsory bytes) and the bf16
    tensor peak (its useful flops); the per-chunk gradient kernel, which reads and
    writes almost all of those bytes, reported beside it.  `with_forward_outputs`: a
    training step, which also writes the forward's o and ht (its flops, the forward's
    once, are already counted: the backward's own recompute is skipped)."""
    r, wr = chunk_bwd_bytes(inp)
    if with_forward_outputs:
        w = inp["workload"]
        wr += _nbytes(inp["v"]) + inp["N"] * w.HV * w.K * w.V * 4
    flops = chunk_bwd_flops(inp)
    t_hbm = (r + wr) / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    sec = ms / 1e3
    unit_ms = sum(t for n, (t, _) in per_kernel.items() if n.startswith("chunk_bwd_unit")) / prof_steps
    out = {"kernel": ("kda_chunk_fwd_save + kda_chunk_bwd (all launches)" if with_forward_outputs
                      else "kda_chunk_bwd (all launches)"), "kernel_ms": ms,
           "hbm": {"achieved": (r + wr) / sec / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                   "frac": (r + wr) / sec / 1e9 / peaks["hbm_gbs"], "algorithmic_bytes": r + wr},
           "tensor": {"achieved": flops / sec / 1e12, "peak": peaks["bf16_tflops"],
                      "unit": "TFLOP/s", "frac": flops / sec / 1e12 / peaks["bf16_tflops"],
                      "algorithmic_flops": flops},
           "unit_kernel": {"ms": unit_ms,
                           "gbs": (r + wr - _nbytes(inp["h0"])) / (unit_ms / 1e3) / 1e9
                           if unit_ms > 0 else None},
           "peak_source": peaks["source"], "traffic": _traffic("chunk_bwd_unit_tc", name)}
    top = out["hbm"] if t_hbm >= t_tc else out["tensor"]
    out.update({"bound": "hbm" if t_hbm >= t_tc else "tensor", "achieved": top["achieved"],
                "peak": top["peak"], "unit": top["unit"], "frac": top["frac"]})
    return out


def recurrent_flops(inp):
    """fp32 flops of the token recurrence: per (token, value head) two K x V
    reductions over the old state (2 flops per element each) and the decayed
    rank-1 update (a multiply and an FMA per element): 7 K V."""
    w = inp["workload"]
    return 7 * inp["tokens"] * w.HV * w.K * w.V


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


def _traffic(kernel, workload="train"):
    """dram bytes per step (all the kernel's launches in one call) from the
    committed ncu summary, if it was taken on the current source of that kernel
    for this workload; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    rec = table.get(f"{kernel}@{workload}") or table.get(kernel)
    if not rec or rec.get("bench_workload", "train") != workload:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    if digest != rec.get("source_sha256_16"):
        return None
    return rec["dram_bytes_per_step"]


def workload_config(name, world=1):
    """The `config` of a bench line, from the workload's definition alone, so
    both arms (ours and the reference) report the same keys and values."""
    import kda_synth

    idx, over, _, _ = WORKLOADS[name]
    w = kda_synth.workload(idx, **over)
    recurrent = name in RECURRENT
    if w.packed:
        # the packed layout is drawn from the seed: count its sequences and tokens
        offs = kda_synth.make_inputs(kda_synth.workload(w, B=1, T=1, H=1, HV=1, K=1, V=1,
                                                        fill_limit=w.fill_limit,
                                                        len_max=w.len_max),
                                     "cpu")
        seqs, tokens = offs["N"], offs["tokens"]
    else:
        seqs, tokens = w.B, w.B * w.T
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.HV, "K": w.K, "V": w.V,
            "input_dtype": "bf16" if w.dtype == _bf16() else "f32", "gate_dtype": "f32",
            "gate": f"-U({w.g_lo:g},{w.g_hi:g}) log2 per token",
            "h0": "N(0,0.1) fp32" if w.has_h0 else "none",
            "ht": "in place (ht == h0)" if recurrent else "stored",
            "pass": "backward" if name in BACKWARD else "forward",
            "sequences": seqs, "tokens": tokens,
            "l2_flush": "512 MiB write between timed steps",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def _bf16():
    import torch

    return torch.bfloat16


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(inp, max_tokens):
    """The first sequences (or, for one long sequence, the first tokens) of the
    workload, up to about `max_tokens` tokens, sliced where the inputs live and
    then copied to the host.  Returns (inputs for oracle.recurrent, tokens, text)."""
    q, k, v, g, beta, h0, cu = (inp[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    B, T = q.shape[0], q.shape[1]
    if cu is not None:
        offs = cu.cpu().tolist()
        s = 1
        while s < len(offs) - 1 and (offs[s + 1] <= max_tokens or offs[s] == 0):
            s += 1
        L = offs[s]
        part = dict(q=q[:, :L], k=k[:, :L], v=v[:, :L], g=g[:, :L], beta=beta[:, :L],
                    h0=None if h0 is None else h0[:s], cu_seqlens=cu[: s + 1])
        text = f"first {s} of {len(offs) - 1} sequence slots ({L} tokens)"
    else:
        nb = max(1, min(B, max_tokens // T))
        L = min(T, max(1, max_tokens)) if nb == 1 else T
        part = dict(q=q[:nb, :L], k=k[:nb, :L], v=v[:nb, :L], g=g[:nb, :L], beta=beta[:nb, :L],
                    h0=None if h0 is None else h0[:nb], cu_seqlens=None)
        L = nb * L
        text = (f"first {nb} of {B} sequences" if nb > 1 or B > 1 else "sequence") + \
            f", {L} tokens"
    part = {n: (None if t is None else t.cpu()) for n, t in part.items()}
    return part, L, text


def _oracle_run(part):
    import oracle

    if "dout" in part:  # a backward workload: the fp64 chunk-form gradients
        from oracle import chunk_backward

        f64 = lambda t: None if t is None else t.double().numpy()
        chunk_backward.chunk_grads(f64(part["q"]), f64(part["k"]), f64(part["v"]), f64(part["g"]),
                                   f64(part["beta"]), f64(part["dout"]), f64(part["h0"]),
                                   f64(part["dht"]),
                                   cu_seqlens=None if part["cu_seqlens"] is None
                                   else part["cu_seqlens"].numpy())
        return
    oracle.recurrent(part["q"], part["k"], part["v"], part["g"], part["beta"], h0=part["h0"],
                     cu_seqlens=part["cu_seqlens"])


def _with_grads_in(part):
    """A backward sample's dL/do and dL/dht, drawn once from a fixed seed."""
    import torch

    gen = torch.Generator().manual_seed(11)
    v, q = part["v"], part["q"]
    n = q.shape[0] if part["cu_seqlens"] is None else part["cu_seqlens"].numel() - 1
    part = dict(part)
    part["dout"] = torch.randn(v.shape, generator=gen).to(v.dtype)
    part["dht"] = torch.randn(n, v.shape[2], q.shape[3], v.shape[3], generator=gen)
    return part


def cpu_oracle_rate(inp, budget_s=10.0, max_runs=3):
    """Oracle tokens/s on a bounded sample of the workload sized to ~budget_s of
    CPU work (all value heads of the sampled sequences)."""
    import oracle

    probe, pL, _ = oracle_sample(inp, 64)
    t0 = time.perf_counter()
    _oracle_run(probe)  # also loads the library
    t0 = time.perf_counter()
    _oracle_run(probe)
    probe_rate = pL / max(1e-6, time.perf_counter() - t0)
    part, L, text = oracle_sample(inp, int(max(64, probe_rate * budget_s / max_runs)))
    runs, t_total = 0, 0.0
    while runs < max_runs and (t_total < budget_s or runs == 0):
        t0 = time.perf_counter()
        _oracle_run(part)
        t_total += time.perf_counter() - t0
        runs += 1
    return L * runs / t_total, runs, text, oracle.num_threads()


def run_reference(args):
    """The oracle as the reference arm: each step one bounded sample."""
    import torch  # noqa: F401

    rank = _env_int("RANK", 0)
    if rank != 0:
        return 0
    if args.workload in RECURRENT:
        # The same distributions drawn for 64 sequences: the sample never needs more.
        import kda_synth

        idx, over, _, _ = WORKLOADS[args.workload]
        inp = kda_synth.make_inputs(kda_synth.workload(idx, **over, B=64, decode_seqs=64), "cpu")
    else:
        inp = _make_inputs(args.workload, "cpu")
    w = inp["workload"]
    backward = args.workload in BACKWARD
    # Size a step so that warm-up + steps end within ~2 minutes.
    probe, pL, _ = oracle_sample(inp, 256)
    if backward:
        probe = _with_grads_in(probe)
    _oracle_run(probe)
    t0 = time.perf_counter()
    _oracle_run(probe)
    probe_rate = pL / max(1e-6, time.perf_counter() - t0)
    per_step_s = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    part, L, text = oracle_sample(inp, int(max(16, probe_rate * per_step_s)))
    if backward:
        part = _with_grads_in(part)
    import oracle

    for _ in range(args.warmup):
        _oracle_run(part)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_run(part)
    dt = time.perf_counter() - t0
    ms = 1e3 * dt / max(1, args.steps)
    value = L / (ms / 1e3)
    line = {
        "impl": "reference", "metric": _metric(args.workload, w), "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(args.workload, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT,
                         "cores": 1 if backward else oracle.num_threads(),
                         "kind": "oracle", "sample_tokens_per_step": L,
                         "sample": f"{text}, all {w.HV} heads, per step" +
                                   (" (fp64 chunk-form gradients, numpy)" if backward else "")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ ours
def run_ours(args):
    import torch

    import gated_delta_rule_cumsum_gb300 as kda

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

    inp = _make_inputs(args.workload, dev)
    w = inp["workload"]
    recurrent = args.workload in RECURRENT
    q, k, v, g, beta, h0, cu = (inp[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    shape = kda.make_shape(q, v, cu)
    o = torch.empty_like(v)
    status = kda.new_status(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    backward = args.workload in BACKWARD
    chunk_bwd = args.workload in CHUNK_BWD
    if backward:
        # dL/do and dL/dht drawn once; the gradients land in preallocated fp32 buffers.
        gen = torch.Generator(device=dev).manual_seed(11)
        dout = torch.randn(v.shape, generator=gen, device=dev).to(q.dtype)
        ht = torch.randn(inp["N"], w.HV, w.K, w.V, generator=gen, device=dev)  # dht
        ws_bytes = (kda.kda_chunk_bwd_workspace_size(shape) if chunk_bwd
                    else kda.kda_recurrent_bwd_workspace_size(shape))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        grads = [torch.empty(t.shape, dtype=torch.float32, device=dev) for t in (q, k, v, g, beta)]
        dh0 = torch.empty(inp["N"], w.HV, w.K, w.V, dtype=torch.float32, device=dev)
        bwd_call = kda.kda_chunk_bwd if chunk_bwd else kda.kda_recurrent_bwd
        if args.workload == "train_step":
            o_fwd = torch.empty_like(v)
            ht_fwd = torch.empty(inp["N"], w.HV, w.K, w.V, dtype=torch.float32, device=dev)
            shape_saved = kda.make_shape(q, v, cu, flags=kda.KDA_FLAG_BWD_SAVED)

            def call(q_, k_, v_, g_, beta_, h0_, o_, ht_, st):
                kda.kda_chunk_fwd_save(q_, k_, v_, g_, beta_, h0_, cu, shape, None, o_fwd, ht_fwd,
                                       ws, status, st)
                kda.kda_chunk_bwd(q_, k_, v_, g_, beta_, h0_, cu, shape_saved, o_, ht_, *grads,
                                  dh0, ws, status, st)
        else:
            def call(q_, k_, v_, g_, beta_, h0_, o_, ht_, st):
                bwd_call(q_, k_, v_, g_, beta_, h0_, cu, shape, o_, ht_, *grads, dh0, ws, status,
                         st)
        o = dout
    elif recurrent:
        # Decode keeps the state resident and updates it in place (ht == h0).
        ht, ws = h0, None

        def call(q_, k_, v_, g_, beta_, h0_, o_, ht_, st):
            kda.kda_recurrent_fwd(q_, k_, v_, g_, beta_, h0_, cu, shape, o_, ht_, status, st)
    else:
        ht = torch.empty(inp["N"], w.HV, w.K, w.V, dtype=torch.float32, device=dev)
        ws = torch.empty(kda.kda_chunk_workspace_size(shape), dtype=torch.uint8, device=dev)

        def call(q_, k_, v_, g_, beta_, h0_, o_, ht_, st):
            kda.kda_chunk_fwd(q_, k_, v_, g_, beta_, h0_, cu, shape, o_, ht_, ws, status, st)

    def step():
        call(q, k, v, g, beta, h0, o, ht, stream)

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
    # The dominant kernel and its device time per step: a pipelined call launches
    # the prep and the scan twice each (two parts of every sequence), so the
    # compulsory bytes of a step are set against the kernel's time per step.
    dom = max(per_kernel, key=lambda n: per_kernel[n][0])
    dom_ms = per_kernel[dom][0] / prof_steps
    peaks = _peaks()
    dom_bytes = kernel_algorithmic_bytes(dom, inp)
    traffic = _traffic(dom, args.workload)
    r_b, w_b = algorithmic_bytes(inp)
    path_gbs = (r_b + w_b) / (ms / 1e3) / 1e9
    if (backward and not chunk_bwd) or args.workload.startswith("prefill"):
        # the fp32-bound kernels' denominator, measured here by an FMA-loop kernel
        peak = kda.kda_measure_fp32_fma_peak(stream)
        peak_source = ("measured in this run: FMA-loop microbenchmark "
                       "(kda_measure_fp32_fma_peak, 16 chains x 8x256 threads per SM)")
    if chunk_bwd:
        roofline = chunk_bwd_roofline(inp, per_kernel, prof_steps, ms, peaks, args.workload,
                                      with_forward_outputs=args.workload == "train_step")
    elif backward:
        flops = BWD_FLOPS_PER_ELEMENT * inp["tokens"] * w.HV * w.K * w.V
        step_ms = sum(t for t, _ in per_kernel.values()) / prof_steps
        roofline = {"bound": "alu", "kernel": "recurrent_ckpt+recurrent_bwd",
                    "achieved": flops / (step_ms / 1e3) / 1e12, "peak": peak, "unit": "TFLOP/s",
                    "frac": flops / (step_ms / 1e3) / 1e12 / peak, "traffic": None,
                    "algorithmic_flops": flops, "kernel_ms": step_ms,
                    "peak_source": peak_source,
                    "nominal_peak": fp32_fma_tflops(torch.cuda.get_device_properties(dev)
                                                    .multi_processor_count, peaks["sm_max_mhz"])}
    elif args.workload.startswith("prefill"):
        # 256 tokens per state: the recurrence's fp32 FMAs, not HBM, bound it.
        flops = recurrent_flops(inp)
        roofline = {"bound": "alu", "kernel": dom, "achieved": flops / (dom_ms / 1e3) / 1e12,
                    "peak": peak, "unit": "TFLOP/s",
                    "frac": flops / (dom_ms / 1e3) / 1e12 / peak, "traffic": traffic,
                    "algorithmic_flops": flops, "kernel_ms": dom_ms,
                    "peak_source": peak_source,
                    "nominal_peak": fp32_fma_tflops(torch.cuda.get_device_properties(dev)
                                                    .multi_processor_count, peaks["sm_max_mhz"])}
    else:
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "traffic": traffic, "algorithmic_bytes": dom_bytes,
                    "kernel_ms": dom_ms, "peak_source": peaks["source"],
                    "path_gbs": path_gbs, "path_frac": path_gbs / peaks["hbm_gbs"]}

    # End to end through the C ABI with host buffers: every step copies its inputs
    # from pinned host memory, runs the call and reads the results back (o and the
    # final state; decode's state stays resident and is updated in place, so only
    # o comes back).  Pipelined: step i's H2D (copy stream) overlaps step i-1's
    # call (compute stream) and step i-2's D2H (copy-back stream), with two sets
    # of device inputs and outputs; events order each buffer's reuse.  The
    # one-stream sequential time is reported beside it.
    names = ("q", "k", "v", "g", "beta") + (("h0",) if h0 is not None and not recurrent else ())
    h2d = sum(_nbytes(inp[n]) for n in names)
    e2e = None
    if backward:
        e2e = {"value": None, "unit": UNIT,
               "skipped": "backward: in training the gradients stay on the device"}
    elif h2d > E2E_MAX_H2D:
        e2e = {"value": None, "unit": UNIT,
               "skipped": f"{h2d / 2**30:.1f} GiB of inputs per step exceed the "
                          f"{E2E_MAX_H2D >> 30} GiB pinned staging limit"}
    else:
        host = {n: inp[n].cpu().pin_memory() for n in names}
        dev_in = [{n: torch.empty_like(inp[n]) for n in names} for _ in range(2)]
        dev_o = [torch.empty_like(o) for _ in range(2)]
        dev_ht = [ht, ht] if recurrent else [torch.empty_like(ht) for _ in range(2)]
        o_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
        ht_h = None if recurrent else \
            [torch.empty(ht.shape, dtype=ht.dtype, pin_memory=True) for _ in range(2)]
        d2h = _nbytes(o_h[0]) + (0 if recurrent else _nbytes(ht_h[0]))
        e2e_steps = min(args.steps, 30)
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_comp = torch.cuda.Stream(dev)

        def run_call(j, st):
            d = dev_in[j]
            call(d["q"], d["k"], d["v"], d["g"], d["beta"], d.get("h0", h0), dev_o[j], dev_ht[j],
                 st)

        def read_back(j):
            o_h[j].copy_(dev_o[j], non_blocking=True)
            if ht_h is not None:
                ht_h[j].copy_(dev_ht[j], non_blocking=True)

        def run_pipeline(nsteps):
            up_done = [torch.cuda.Event() for _ in range(nsteps)]
            comp_done = [torch.cuda.Event() for _ in range(nsteps)]
            down_done = [torch.cuda.Event() for _ in range(nsteps)]
            for i in range(nsteps):
                j = i % 2
                with torch.cuda.stream(s_up):
                    if i >= 2:
                        s_up.wait_event(comp_done[i - 2])  # buffer j's previous call read it
                    for n in names:
                        dev_in[j][n].copy_(host[n], non_blocking=True)
                    up_done[i].record(s_up)
                s_comp.wait_event(up_done[i])
                if i >= 2:
                    s_comp.wait_event(down_done[i - 2])  # outputs j have been read back
                run_call(j, s_comp)
                comp_done[i].record(s_comp)
                with torch.cuda.stream(s_down):
                    s_down.wait_event(comp_done[i])
                    read_back(j)
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
            for n in names:
                dev_in[0][n].copy_(host[n], non_blocking=True)
            run_call(0, stream)
            read_back(0)

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
        e2e = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "mode": "pipelined: step i's H2D overlaps step i-1's call and step i-2's D2H "
                       "(two buffer sets, three streams; wall clock over the steps)",
               "sequential_ms_per_step": e2e_seq_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not backward:
        rate, runs, text, cores = cpu_oracle_rate(inp, budget_s=10.0)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{text} x {w.HV} heads, {runs} run(s), fp64"}

    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    # bf16 operands with fp32 accumulation on the tensor-core path; fp32 on the SIMT path
    compute_dtype = "bf16" if any(n.endswith("_tc") for n in per_kernel) else "f32"
    line = {
        "metric": _metric(args.workload, w), "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": compute_dtype, "data": "synthetic",
        "config": workload_config(args.workload, world),
        "roofline": roofline,
        "kernels": {n: {"ms_per_launch": t / c, "launches_per_step": c / prof_steps}
                    for n, (t, c) in per_kernel.items()},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="train")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    _, _, d_steps, d_warm = WORKLOADS[args.workload]
    if args.steps is None:
        args.steps = d_steps
    if args.warmup is None:
        args.warmup = d_warm
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
