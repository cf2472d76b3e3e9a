"""Seeded synthetic inputs for the KDA forward workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so the oracle and the CUDA path can both take their inputs
from it.  Recipe (fixed draw order: q, k, v, beta-logits, g, h0, then sequence
lengths and empty-slot positions):

* q, k ~ N(0, 1) in fp32, each row L2-normalised over K (the data recipe of the
  workloads, not the op's in-kernel flag), then cast to the workload dtype;
* v ~ N(0, 1); beta = sigmoid(N(0, 1)); g = -Uniform(lo, hi) per token and
  channel (base-2 log decay, fp32); h0 ~ N(0, 0.1^2) fp32 where present;
* packed workloads: sequence lengths ~ Geometric(p) on {1, 2, ...}, clipped and
  redrawn until they fit, empty slots (repeated offsets) inserted at seeded
  positions, rows at or beyond the terminal offset filled with NaN.

Small workloads are drawn with a CPU generator (bit-identical on every host).
The decode workload's multi-GB state is drawn on the target device with a
device generator; parity checks copy the sampled slices they need back to the
host.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "workload"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int                     # physical rows per batch entry (capacity when packed)
    H: int
    HV: int
    K: int
    V: int
    dtype: torch.dtype         # q, k, v, beta (and o)
    g_lo: float
    g_hi: float
    has_h0: bool
    seed: int
    packed: bool = False
    n_seqs: int = 0            # non-empty sequences when packed
    n_empty: int = 0           # empty slots when packed
    geo_p: float = 0.0
    len_max: int = 0
    fill_limit: int = 0        # sum of lengths must stay <= this
    decode_seqs: int = 0       # >0: one sequence per slot, `T` tokens each
    device_rng: bool = False   # draw on the target device

    @property
    def tokens_upper(self) -> int:
        return self.B * self.T


# The five workloads (tiny, training shape, grouped value heads, packed varlen,
# decode).  Seeds: the tiny workload uses 0, the others their index.
WORKLOADS = {
    0: Workload("tiny_fp32_B1_T128_H1_K64_V64", 1, 128, 1, 1, 64, 64, torch.float32,
                0.01, 0.5, True, 0),
    1: Workload("train_bf16_B1_T8192_H16_HV16_K128_V128", 1, 8192, 16, 16, 128, 128,
                torch.bfloat16, 0.001, 0.3, False, 1),
    2: Workload("gva_bf16_B4_T4096_H8_HV32_K128_V128", 4, 4096, 8, 32, 128, 128,
                torch.bfloat16, 0.001, 0.3, True, 2),
    3: Workload("packed_bf16_N72_Tcap32768_H32_HV32_K128_V128", 1, 32768, 32, 32, 128, 128,
                torch.bfloat16, 0.001, 0.3, True, 3, packed=True, n_seqs=64, n_empty=8,
                geo_p=1.0 / 512, len_max=4096, fill_limit=32704),
    4: Workload("decode_bf16_N4096_T1_H32_HV32_K128_V128", 4096, 1, 32, 32, 128, 128,
                torch.bfloat16, 0.001, 0.3, True, 4, decode_seqs=4096, device_rng=True),
}


def workload(idx_or_name, **overrides) -> Workload:
    """Look up a workload by index or name; keyword overrides give variants
    (e.g. the 256-token prefill variant of the decode workload: T=256)."""
    if isinstance(idx_or_name, Workload):
        w = idx_or_name
    elif isinstance(idx_or_name, int):
        w = WORKLOADS[idx_or_name]
    else:
        w = next(x for x in WORKLOADS.values() if x.name == idx_or_name)
    if overrides:
        w = dataclasses.replace(w, **overrides)
    return w


def _normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _uniform(shape, gen, device):
    return torch.rand(shape, generator=gen, device=device, dtype=torch.float32)


def _rownorm(x):
    return x / x.square().sum(-1, keepdim=True).sqrt()


def _packed_layout(w: Workload, gen) -> list:
    """Offsets [N+1] with `n_empty` repeated offsets at seeded positions."""
    while True:
        u = _uniform((w.n_seqs,), gen, "cpu").double().clamp_min(1e-300)
        lens = torch.floor(torch.log(u) / math.log1p(-w.geo_p)).long() + 1
        lens = lens.clamp(1, w.len_max)
        if int(lens.sum()) <= w.fill_limit:
            break
    n_slots = w.n_seqs + w.n_empty
    empty_pos = set(torch.randperm(n_slots, generator=gen)[: w.n_empty].tolist())
    offsets, it, pos = [0], iter(lens.tolist()), 0
    for s in range(n_slots):
        pos += 0 if s in empty_pos else next(it)
        offsets.append(pos)
    return offsets


def make_inputs(w, device="cpu", seed: Optional[int] = None, packed_decode: bool = False):
    """Draw one workload's inputs.

    Returns a dict with q, k, v, g, beta, h0 (or None), cu_seqlens (int32 or None),
    and `N` (number of state slots), `tokens` (valid tokens), `workload`.
    `packed_decode=True` lays the decode workload out as one packed row with
    cu_seqlens = arange(N+1)*T instead of a dense batch.
    """
    w = workload(w)
    seed = w.seed if seed is None else seed
    dev = torch.device(device)
    gdev = dev if w.device_rng else torch.device("cpu")
    gen = torch.Generator(device=gdev)
    gen.manual_seed(seed)

    B, T = w.B, w.T
    if w.decode_seqs and packed_decode:
        B, T = 1, w.decode_seqs * w.T
    q = _rownorm(_normal((B, T, w.H, w.K), gen, gdev))
    k = _rownorm(_normal((B, T, w.H, w.K), gen, gdev))
    v = _normal((B, T, w.HV, w.V), gen, gdev)
    beta = torch.sigmoid(_normal((B, T, w.HV), gen, gdev))
    g = -(w.g_lo + (w.g_hi - w.g_lo) * _uniform((B, T, w.HV, w.K), gen, gdev))

    cu = None
    if w.packed:
        offsets = _packed_layout(w, torch.Generator().manual_seed(seed + 7919))
        N = len(offsets) - 1
        cu = torch.tensor(offsets, dtype=torch.int32)
        end = offsets[-1]
        for t in (q, k, v, g, beta):
            t[:, end:] = float("nan")
    elif w.decode_seqs and packed_decode:
        N = w.decode_seqs
        cu = torch.arange(N + 1, dtype=torch.int32) * w.T
    else:
        N = B
    h0 = None
    if w.has_h0:
        h0 = 0.1 * _normal((N, w.HV, w.K, w.V), gen, gdev)

    tokens = int(cu[-1]) if cu is not None else B * T
    out = dict(q=q.to(w.dtype), k=k.to(w.dtype), v=v.to(w.dtype), beta=beta.to(w.dtype),
               g=g, h0=h0, cu_seqlens=cu, N=N, tokens=tokens, workload=w)
    for name in ("q", "k", "v", "beta", "g", "h0", "cu_seqlens"):
        if out[name] is not None:
            out[name] = out[name].to(dev).contiguous()
    return out
