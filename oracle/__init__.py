"""fp64 CPU oracle for the KDA forward -- TEST INFRASTRUCTURE ONLY.

Only tests/, `__graft_entry__.smoke()` and the `cpu_baseline` / reference leg of
bench.py may import this package.  The product (the CUDA library and its Python
binding) never imports it and has no CPU fallback.

Two independent formulations live here:

* `recurrent` / `gate_cumsum` -- the C library `kda_oracle.c`: the token-by-token
  recurrence of the gated delta rule with per-channel decay, exactly as defined
  in attention-gym PR #317 ("Add fused recurrent_kda for decode and inference
  prefill", PR description) and the conventions of kernel-fun 0.2.0.dev1 sdist,
  ALGORITHM.md (preamble), plus the chunk-local gate cumsum of ALGORITHM.md
  "Stage 1 -- cumsum".
* `chunk_form.chunk_forward` -- the chunked (WY / UT-transform) formulation of
  ALGORITHM.md "Stage 1" through "Stage 3+4", in numpy fp64.
* `backward.recurrent_grads` -- the gradients (dq, dk, dv, dg, dbeta, dh0) of the
  token recurrence (kernel-fun 0.2.0.dev1 sdist, ALGORITHM.md, "Backward"), in
  PyTorch fp64 by reverse mode; pinned in tests/test_oracle_backward.py against
  finite differences of the C recurrence.
* `chunk_backward.chunk_grads` -- the same gradients by the chunk form, stage by
  stage in the order of ALGORITHM.md, "Backward" (recompute, re-scan, dAv, dhu,
  wy_dqkg, intra, dg cumsum), in numpy fp64, with the per-chunk intermediates on
  request and the L2-norm and activation options; pinned in
  tests/test_oracle_chunk_backward.py against `backward`.
* `activation` -- the optional input activations (gate -exp(A_log) softplus(g +
  dt_bias), beta sigmoid) of kernel-fun 0.2.0.dev1 wheel, kda/chain.py and
  kda/ops.py, in numpy fp64; pinned in tests/test_oracle_activation.py.

Each pins the other (tests/test_oracle_pins.py), beside closed forms, invariants
and brute force that the pages and the mathematics fix.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np

from .build import build_oracle

__all__ = ["recurrent", "gate_cumsum", "num_threads", "lib"]

_LIB = None


def _bind(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    L.kda_oracle_recurrent.argtypes = [dp, dp, dp, dp, dp, dp, ip] + [ctypes.c_int] * 7 + [
        ctypes.c_double, ctypes.c_double, ctypes.c_int, dp, dp]
    L.kda_oracle_recurrent.restype = ctypes.c_int
    L.kda_oracle_gate_cumsum.argtypes = [dp, ip] + [ctypes.c_int] * 6 + [ctypes.c_double, dp]
    L.kda_oracle_gate_cumsum.restype = ctypes.c_int
    L.kda_oracle_num_threads.argtypes = []
    L.kda_oracle_num_threads.restype = ctypes.c_int
    return L


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = _bind(build_oracle())
    return _LIB


def num_threads() -> int:
    """Host threads the oracle's OpenMP loops use."""
    return int(lib().kda_oracle_num_threads())


def _f64(x) -> np.ndarray:
    """Exact upcast to a C-contiguous float64 array (bf16 and fp32 embed exactly)."""
    if x is None:
        return None
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if x is None:
        return None
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu").numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _dptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_int32)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def recurrent(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, g_scale=1.0,
              l2norm=False, o_fill=float("nan"), want_state=True, _library=None):
    """Token-by-token fp64 recurrence.  Returns (o, ht) as float64 numpy arrays.

    Shapes: q, k [B,T,H,K]; v [B,T,HV,V]; g [B,T,HV,K]; beta [B,T,HV];
    h0 [N,HV,K,V] or None; cu_seqlens [N+1] int32 or None (then N = B).
    `scale=None` means K^-1/2 (kernel-fun 0.2.0.dev1 wheel, kda/ops.py, chunk_kda).
    Rows of o outside every sequence keep `o_fill`.
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    h0 = _f64(h0)
    cu = _i32(cu_seqlens)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = B if cu is None else cu.shape[0] - 1
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    o = np.full((B, T, HV, V), o_fill, dtype=np.float64)
    ht = np.zeros((N, HV, K, V), dtype=np.float64) if want_state else None
    rc = (_library or lib()).kda_oracle_recurrent(
        _dptr(q), _dptr(k), _dptr(v), _dptr(g), _dptr(beta), _dptr(h0), _iptr(cu),
        B, T, H, HV, K, V, N, float(scale), float(g_scale), int(bool(l2norm)),
        _dptr(o), _dptr(ht))
    if rc != 0:
        raise ValueError(f"kda_oracle_recurrent failed with code {rc}")
    return o, ht


def gate_cumsum(g, cu_seqlens=None, chunk=64, g_scale=1.0, fill=float("nan"), _library=None):
    """Chunk-local inclusive cumsum of g (times g_scale) in fp64; [B,T,HV,K]."""
    g = _f64(g)
    cu = _i32(cu_seqlens)
    B, T, HV, K = g.shape
    N = B if cu is None else cu.shape[0] - 1
    out = np.full(g.shape, fill, dtype=np.float64)
    rc = (_library or lib()).kda_oracle_gate_cumsum(_dptr(g), _iptr(cu), B, T, HV, K, N, int(chunk),
                                      float(g_scale), _dptr(out))
    if rc != 0:
        raise ValueError(f"kda_oracle_gate_cumsum failed with code {rc}")
    return out
