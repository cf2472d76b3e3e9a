"""fp64 gradients of the KDA token recurrence -- TEST INFRASTRUCTURE ONLY.

The backward's contract is that of kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md,
"Backward", and of kernel-fun 0.2.0.dev1 wheel, kda/chain.py, `backward`: given
the output gradient do and the final-state gradient dht it returns dq, dk, dv,
dbeta, dg and dh0, where dg is taken with respect to the per-token decay (the
gate before any cumsum) and dq / dk are summed over the value heads that share a
q/k head.  The method reaches the result of the token recurrence, so the
gradients are those of the plain recurrence (attention-gym PR #317, PR
description; the same definition the C oracle in this package integrates):

    S_t = Diag(2^(g_scale g_t)) S_{t-1}
    delta_t = beta_t (v_t - S_t^T k_t)      (S_t here: after the decay)
    S_t = S_t + k_t delta_t^T
    o_t = scale S_t^T q_t

written out once more below in PyTorch fp64 and differentiated by PyTorch's
reverse mode (a library primitive standing for the chain rule).  The loss whose
gradients are returned is  sum(o * do) + sum(ht * dht).  tests/test_oracle_backward.py
pins it against central finite differences of the C oracle's forward (an
independent implementation) and against the closed form at beta = 0.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["recurrent_grads"]


def recurrent_grads(q, k, v, g, beta, do, h0=None, dht=None, cu_seqlens=None, scale=None,
                    g_scale=1.0, l2norm=False, A_log=None, dt_bias=None, beta_scale=0.0,
                    beta_bf16=False):
    """Gradients of sum(o * do) + sum(ht * dht) of the token recurrence, in fp64.
    With `l2norm` the recurrence uses q / sqrt(sum q^2 + 1e-6) and the same of k per
    (token, head) (kernel-fun 0.2.0.dev1 wheel, kda/autograd.py, l2norm option), and
    the gradients are those of the raw q and k.
    With `A_log` the gate is raw: the recurrence uses -exp(A_log[hv]) softplus(g +
    dt_bias[hv, d]) (natural log, times g_scale), and with `beta_scale` > 0 beta is
    raw too: sigmoid(beta) * beta_scale (kernel-fun 0.2.0.dev1 wheel, kda/chain.py,
    gate_cumsum and gate_backward; kda/ops.py, chunk_kda), rounded to bf16 in value
    when `beta_bf16` (the rounding passes gradients straight through).  The
    gradients are then those of the raw g and beta, plus dA_log [HV] and dt_bias's.

    Shapes: q, k [B,T,H,K]; v, do [B,T,HV,V]; g [B,T,HV,K] (per-token log2 decay);
    beta [B,T,HV]; h0, dht [N,HV,K,V] or None; cu_seqlens [N+1] or None (then N = B).
    Returns a dict of float64 numpy arrays dq, dk, dv, dg, dbeta, dh0 (dh0 None when
    h0 is None).  Rows outside every sequence get zero gradients.
    """
    import torch

    def leaf(x):
        return torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True)

    q, k, v, g, beta = (leaf(x) for x in (q, k, v, g, beta))
    A_log_t = None if A_log is None else leaf(A_log)
    dt_t = None if dt_bias is None else leaf(dt_bias)
    do = torch.tensor(np.asarray(do, dtype=np.float64))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    cu = None if cu_seqlens is None else [int(x) for x in np.asarray(cu_seqlens)]
    N = B if cu is None else len(cu) - 1
    h0t = None if h0 is None else leaf(h0)
    dhtt = None if dht is None else torch.tensor(np.asarray(dht, dtype=np.float64))
    if scale is None:
        scale = 1.0 / math.sqrt(K)

    loss = torch.zeros((), dtype=torch.float64)
    for n in range(N):
        b, bos, eos = (n, 0, T) if cu is None else (0, cu[n], cu[n + 1])
        S = h0t[n] if h0t is not None else torch.zeros(HV, K, V, dtype=torch.float64)
        for t in range(bos, eos):
            qr, kr = q[b, t], k[b, t]                           # [H, K]
            if l2norm:
                qr = qr / torch.sqrt((qr * qr).sum(-1, keepdim=True) + 1e-6)
                kr = kr / torch.sqrt((kr * kr).sum(-1, keepdim=True) + 1e-6)
            qt = qr.repeat_interleave(G, dim=0)                 # [HV, K]
            kt = kr.repeat_interleave(G, dim=0)
            gt, bt = g[b, t], beta[b, t]
            if A_log_t is not None:
                x = gt if dt_t is None else gt + dt_t
                gt = -torch.exp(A_log_t)[:, None] * torch.nn.functional.softplus(x)
            if beta_scale > 0:
                bt = torch.sigmoid(bt) * beta_scale
                if beta_bf16:
                    bt = bt + (bt.to(torch.bfloat16).to(torch.float64) - bt).detach()
            S = torch.exp2(g_scale * gt)[:, :, None] * S  # decay rows
            a = torch.einsum("hkv,hk->hv", S, kt)
            delta = bt[:, None] * (v[b, t] - a)
            S = S + kt[:, :, None] * delta[:, None, :]
            loss = loss + (scale * torch.einsum("hkv,hk->hv", S, qt) * do[b, t]).sum()
        if dhtt is not None:
            loss = loss + (S * dhtt[n]).sum()
    loss.backward()

    def grad(x):
        return np.zeros(tuple(x.shape)) if x.grad is None else x.grad.numpy().copy()

    return dict(dq=grad(q), dk=grad(k), dv=grad(v), dg=grad(g), dbeta=grad(beta),
                dh0=None if h0t is None else grad(h0t),
                dA_log=None if A_log_t is None else grad(A_log_t),
                ddt_bias=None if dt_t is None else grad(dt_t))
