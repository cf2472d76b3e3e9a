"""Helpers shared by the GPU parity tests: tolerances, error norms, oracle calls
on sampled slices of a workload."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the forward against the fp64 oracle: max-abs error relative to
# the output's max-abs norm, separately for o and ht.  fp32 inputs: 1e-4;
# bf16 inputs with fp32 accumulation: 2e-2.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def to_np(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rel_err(x, ref) -> float:
    """max|x - ref| / max|ref| (infinity norms); NaN anywhere counts as failure."""
    x, ref = to_np(x), to_np(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if x.size == 0:
        return 0.0
    if not np.all(np.isfinite(x)):
        return float("inf")
    denom = float(np.max(np.abs(ref)))
    return float(np.max(np.abs(x - ref))) / max(denom, 1e-30)


def valid_rows(cu, T):
    """Slice of the physical rows that belong to sequences."""
    if cu is None:
        return slice(0, T)
    return slice(0, int(cu[-1]))


def oracle_forward(inp, *, l2norm=False, g_scale=1.0, scale=None, heads=None, seqs=None):
    """fp64 oracle outputs for a workload dict from kda_synth.make_inputs.

    `heads`: optional list of q/k heads h to evaluate (with their HV/H value
    heads); `seqs`: optional list of sequence slots.  Returns a dict mapping
    (n, hv) -> (o [L, V], ht [K, V]) for the evaluated pairs.
    """
    q, k, v, g, beta, h0, cu = (inp[x] for x in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    B, T, H, K = q.shape
    HV = v.shape[2]
    G = HV // H
    heads = list(range(H)) if heads is None else list(heads)
    N = inp["N"]
    seqs = list(range(N)) if seqs is None else list(seqs)
    cu_l = None if cu is None else [int(x) for x in cu.cpu()]
    out = {}
    for n in seqs:
        if cu_l is None:
            b, a, e = n, 0, T
        else:
            b, a, e = 0, cu_l[n], cu_l[n + 1]
        for h in heads:
            vs = slice(h * G, (h + 1) * G)
            h0s = None if h0 is None else h0[n:n + 1, vs]
            o_n, ht_n = oracle.recurrent(
                q[b:b + 1, a:e, h:h + 1], k[b:b + 1, a:e, h:h + 1], v[b:b + 1, a:e, vs],
                g[b:b + 1, a:e, vs], beta[b:b + 1, a:e, vs], h0=h0s, scale=scale,
                g_scale=g_scale, l2norm=l2norm)
            for j in range(G):
                out[(n, h * G + j)] = (o_n[0, :, j], ht_n[0, j])
    return out


def compare_sampled(inp, o, ht, ref, tol):
    """Largest relative errors of o and ht over the evaluated (n, hv) pairs,
    normalised by the max-abs of the evaluated reference values."""
    cu = inp["cu_seqlens"]
    cu_l = None if cu is None else [int(x) for x in cu.cpu()]
    T = inp["q"].shape[1]
    num_o = num_h = 0.0
    den_o = den_h = 0.0
    for (n, hv), (o_ref, h_ref) in ref.items():
        if cu_l is None:
            o_gpu = o[n, :, hv]
        else:
            o_gpu = o[0, cu_l[n]:cu_l[n + 1], hv]
        og = to_np(o_gpu)
        if og.size:
            if not np.all(np.isfinite(og)):
                return float("inf"), float("inf")
            num_o = max(num_o, float(np.max(np.abs(og - o_ref))))
            den_o = max(den_o, float(np.max(np.abs(o_ref))))
        if ht is not None:
            hg = to_np(ht[n, hv])
            if not np.all(np.isfinite(hg)):
                return float("inf"), float("inf")
            num_h = max(num_h, float(np.max(np.abs(hg - h_ref))))
            den_h = max(den_h, float(np.max(np.abs(h_ref))))
    e_o = num_o / max(den_o, 1e-30)
    e_h = num_h / max(den_h, 1e-30) if ht is not None else 0.0
    return e_o, e_h
