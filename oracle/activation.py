"""fp64 input activations of the KDA op -- TEST INFRASTRUCTURE ONLY (see the
package docstring).

kernel-fun 0.2.0.dev1 wheel, kda/chain.py, gate_cumsum: with use_gate_in_kernel
the op receives the raw gate and owes the natural-log decay
    -exp(A_log) * softplus(g + dt_bias)
before the chunk cumsum, which scales it to log2 by 1/ln 2.  kda/ops.py,
chunk_kda: with use_beta_sigmoid_in_kernel, beta = sigmoid(beta) times 2 when
allow_neg_eigval else 1, then cast to q's dtype.

Readings (the pages give no shapes here): A_log holds one value per value head
[HV], dt_bias one per (value head, channel) [HV, K].  softplus(x) = ln(1 + e^x).
"""
from __future__ import annotations

import numpy as np

from . import _f64


def softplus(x):
    """ln(1 + e^x) in fp64, without overflow."""
    return np.logaddexp(0.0, _f64(x))


def gate(g_raw, A_log, dt_bias=None):
    """Natural-log decay -exp(A_log[hv]) softplus(g_raw + dt_bias[hv, d]) for a
    raw gate [B, T, HV, K]."""
    g = _f64(g_raw)
    a = _f64(A_log)
    x = g if dt_bias is None else g + _f64(dt_bias)[None, None, :, :]
    return -np.exp(a)[None, None, :, None] * softplus(x)


def beta(x, scale, bf16=False):
    """sigmoid(x) * scale in fp64; rounded to bf16 when the op's inputs are bf16."""
    y = scale * 0.5 * (1.0 + np.tanh(0.5 * _f64(x)))  # sigmoid, overflow-free
    if bf16:
        import torch

        y = torch.from_numpy(y).to(torch.bfloat16).to(torch.float64).numpy()
    return y
