"""The chunked (WY / UT-transform) formulation of the KDA forward, numpy fp64.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  This is the second,
independent formulation of the same result: it follows the stage order of
kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, section "Forward", in that page's
notation, per (sequence, value head hv) and per chunk of BT rows:

  Stage 1 -- cumsum:   g2[i] = g_scale * sum_{s <= i in chunk} g[s]   (per channel d)
                       G     = g2[last row of the chunk]
  Stage 2 -- intra/WY: Aqk[i,j] = scale * sum_d q[i,d] k[j,d] 2^(g2[i,d]-g2[j,d]),  i >= j
                       L[i,j]   = beta_i * sum_d k[i,d] k[j,d] 2^(g2[i,d]-g2[j,d]),  i >  j
                       Akk      = (I + L)^-1   (the solved lower-triangular WY inverse,
                                                beta folded in)
                       w  = Akk (beta * 2^g2 * k),   u = Akk (beta * v)
                       kg = k * 2^(G - g2),          qg = q * 2^g2
  Stage 3+4 -- scan:   v' = u - w h
                       o  = scale * qg h + Aqk v'
                       h  = Diag(2^G) h + kg^T v'
                       ht = h after the last chunk.

No blocking beyond the chunk, no factorisation of the exponentials: every
2^(g2_i - g2_j) is formed directly.  The unit lower-triangular inverse uses a
library triangular solve.  A chunk may be shorter than BT (the tail of a
sequence); BT = 1 reduces the scheme to the token recurrence.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.linalg import solve_triangular


def _l2n(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def chunk_sequence(q, k, v, g, beta, h, scale, g_scale=1.0, BT=64):
    """One (sequence, value head): q,k [L,K], v [L,V], g [L,K], beta [L], h [K,V].

    Returns (o [L,V], h_final [K,V]).
    """
    L = q.shape[0]
    V = v.shape[1]
    o = np.empty((L, V), dtype=np.float64)
    h = np.array(h, dtype=np.float64, copy=True)
    for s in range(0, L, BT):
        e = min(s + BT, L)
        qc, kc, vc, bc = q[s:e], k[s:e], v[s:e], beta[s:e]
        n = e - s
        # Stage 1
        g2 = np.cumsum(g_scale * g[s:e], axis=0)          # [n, K]
        G = g2[-1]                                          # [K]
        # Stage 2: the per-dimension gate sits inside both dot products
        rel = np.exp2(g2[:, None, :] - g2[None, :, :])     # [n, n, K]: 2^(g2_i - g2_j)
        qk = np.einsum("id,jd,ijd->ij", qc, kc, rel)
        kk = np.einsum("id,jd,ijd->ij", kc, kc, rel)
        lower_incl = np.tril(np.ones((n, n), dtype=bool))
        strict = np.tril(np.ones((n, n), dtype=bool), k=-1)
        Aqk = np.where(lower_incl, scale * qk, 0.0)
        Lm = np.where(strict, bc[:, None] * kk, 0.0)
        Akk = solve_triangular(np.eye(n) + Lm, np.eye(n), lower=True, unit_diagonal=True)
        w = Akk @ (bc[:, None] * np.exp2(g2) * kc)
        u = Akk @ (bc[:, None] * vc)
        kg = kc * np.exp2(G[None, :] - g2)
        qg = qc * np.exp2(g2)
        # Stage 3+4
        vp = u - w @ h
        o[s:e] = scale * (qg @ h) + Aqk @ vp
        h = np.exp2(G)[:, None] * h + kg.T @ vp
    return o, h


def chunk_forward(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, g_scale=1.0,
                  BT=64, l2norm=False):
    """Whole-call chunked forward with the same layouts and packing rules as
    `oracle.recurrent`.  Inputs: float64 numpy arrays.  Returns (o, ht)."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    group = HV // H
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    if cu_seqlens is None:
        slots = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(x) for x in cu_seqlens]
        slots = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    N = len(slots)
    o = np.full((B, T, HV, V), np.nan)
    ht = np.zeros((N, HV, K, V))
    for n, (b, bos, eos) in enumerate(slots):
        for hv in range(HV):
            hh = hv // group
            h = np.zeros((K, V)) if h0 is None else h0[n, hv]
            if eos == bos:
                ht[n, hv] = h
                continue
            qs, ks = q[b, bos:eos, hh], k[b, bos:eos, hh]
            if l2norm:
                qs, ks = _l2n(qs), _l2n(ks)
            os_, hf = chunk_sequence(qs, ks, v[b, bos:eos, hv], g[b, bos:eos, hv],
                                     beta[b, bos:eos, hv], h, scale, g_scale, BT)
            o[b, bos:eos, hv] = os_
            ht[n, hv] = hf
    return o, ht
