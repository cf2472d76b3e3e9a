"""GB300 (sm_103a) KDA: Python binding over the C ABI of libkda_gb300.so.

Argument marshalling only.  Every step of the forward and the backward runs in the
library's CUDA kernels; torch provides device memory and streams.  There is no CPU
fallback: `load()` raises when the library has not been built.

Binding functions carry the C names (`kda_chunk_fwd`, `kda_recurrent_fwd`,
`kda_gate_cumsum`, `kda_recurrent_bwd`, ...) and take preallocated tensors exactly
like the C calls.  `chunk_kda`, `recurrent_kda`, `gate_cumsum` and
`recurrent_kda_backward` allocate the outputs and call them, mirroring kernel-fun
0.2.0.dev1 wheel, kda/ops.py `chunk_kda` and attention-gym PR #317 `recurrent_kda`;
`kda_autograd` puts them behind torch.autograd.  These run on their tensors'
device (the library launches on the current device and its current stream) and
reject tensors that are not all on one CUDA device.
"""
from __future__ import annotations

import ctypes
import functools
import itertools
import os
from typing import Optional

import torch

__all__ = [
    "KDA_OK", "KDA_ERR_INVALID_ARG", "KDA_ERR_UNSUPPORTED", "KDA_ERR_BAD_CU_SEQLENS",
    "KDA_ERR_CUDA", "KDA_ERR_TIMEOUT", "KDA_FLAG_QK_L2NORM", "KDA_FLAG_G_IS_CUMSUM",
    "KDA_FLAG_SPLIT_SCAN", "KDA_FLAG_SERIAL", "KDA_FLAG_TEST_WAIT_TIMEOUT", "KdaActivation", "make_activation",
    "KdaError", "KdaShape", "load", "library_path", "make_shape",
    "kda_gate_cumsum", "kda_chunk_fwd", "kda_recurrent_fwd", "kda_chunk_workspace_size",
    "kda_workspace_size",
    "kda_recurrent_bwd", "kda_recurrent_bwd_workspace_size", "recurrent_kda_backward", "kda_autograd",
    "kda_chunk_bwd", "kda_chunk_bwd_act", "kda_chunk_bwd_workspace_size", "chunk_kda_backward",
    "kda_chunk_fwd_save", "chunk_kda_forward_save", "KDA_FLAG_BWD_SAVED",
    "kda_gate_cumsum_act", "kda_chunk_fwd_act", "kda_recurrent_fwd_act", "kda_recurrent_bwd_act",
    "kda_chunk_fwd_noalloc", "KDA_NOALLOC_SCRATCH_BYTES",
    "kda_read_device_status", "kda_clear_device_status", "kda_status_string",
    "kda_last_error_message", "kda_version", "kda_profile_enable", "kda_profile_report",
    "kda_profile_reset", "kda_measure_fp32_fma_peak",
    "chunk_kda", "recurrent_kda", "gate_cumsum",
]

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED = 0, 1, 2
KDA_ERR_BAD_CU_SEQLENS, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = 3, 4, 5
KDA_DTYPE_F32, KDA_DTYPE_BF16 = 0, 1
KDA_FLAG_QK_L2NORM, KDA_FLAG_G_IS_CUMSUM, KDA_FLAG_SPLIT_SCAN = 1 << 0, 1 << 1, 1 << 2
KDA_FLAG_SERIAL = 1 << 3
KDA_FLAG_BWD_SAVED = 1 << 4
KDA_FLAG_TEST_WAIT_TIMEOUT = 1 << 31
KDA_DEVICE_BAD_CU_SEQLENS, KDA_DEVICE_TIMEOUT, KDA_DEVICE_INTERNAL = 1 << 0, 1 << 1, 1 << 2
KDA_DEVICE_GATE_RANGE = 1 << 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libkda_gb300.so")
_LIB = None


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED",
                 3: "KDA_ERR_BAD_CU_SEQLENS", 4: "KDA_ERR_CUDA", 5: "KDA_ERR_TIMEOUT"}


class KdaShape(ctypes.Structure):
    """Mirror of `kda_shape` in include/kda.h."""
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("HV", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
                ("num_seqs", ctypes.c_int32), ("dtype", ctypes.c_int),
                ("scale", ctypes.c_float), ("g_scale", ctypes.c_float),
                ("flags", ctypes.c_uint32)]


class KdaActivation(ctypes.Structure):
    """Mirror of `kda_activation` in include/kda.h."""
    _fields_ = [("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("beta_scale", ctypes.c_float)]


def make_activation(A_log=None, dt_bias=None, beta_scale: float = 0.0) -> KdaActivation:
    """A_log [HV] and dt_bias [HV, K] fp32 device tensors (or None); beta_scale 0
    keeps beta as given, 1 or 2 applies sigmoid(beta) * beta_scale."""
    for t, name in ((A_log, "A_log"), (dt_bias, "dt_bias")):
        if t is not None and not t.is_cuda:
            raise KdaError(KDA_ERR_INVALID_ARG, f"{name} must be on a CUDA device")
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous fp32 tensor")
    return KdaActivation(_ptr(A_log), _ptr(dt_bias), float(beta_scale))


def library_path() -> str:
    return _LIB_PATH


# Exported symbols and their signatures (the whole C ABI).
_VP, _SZ, _I32, _ST = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int
_SIGNATURES = {
    "kda_gate_cumsum": (_ST, [_VP, _VP, _VP, ctypes.POINTER(KdaShape), _I32, _VP, _VP]),
    "kda_gate_cumsum_act": (_ST, [_VP, _VP, _VP, ctypes.POINTER(KdaShape),
                                  ctypes.POINTER(KdaActivation), _I32, _VP, _VP]),
    "kda_chunk_fwd_act": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape),
                                ctypes.POINTER(KdaActivation), _VP, _VP, _VP, _SZ, _VP, _VP]),
    "kda_recurrent_fwd_act": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                    ctypes.POINTER(KdaShape), ctypes.POINTER(KdaActivation),
                                    _VP, _VP, _VP, _VP]),
    "kda_chunk_fwd": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape), _VP,
                            _VP, _VP, _SZ, _VP, _VP]),
    "kda_chunk_workspace_size": (_SZ, [ctypes.POINTER(KdaShape)]),
    "kda_workspace_size": (_SZ, [ctypes.POINTER(KdaShape)]),
    "kda_recurrent_bwd": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape),
                                _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "kda_recurrent_bwd_act": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape),
                                    ctypes.POINTER(KdaActivation), _VP, _VP, _VP, _VP, _VP, _VP,
                                    _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "kda_recurrent_bwd_workspace_size": (_SZ, [ctypes.POINTER(KdaShape)]),
    "kda_chunk_bwd": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape),
                            _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "kda_chunk_bwd_workspace_size": (_SZ, [ctypes.POINTER(KdaShape)]),
    "kda_chunk_fwd_save": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape),
                                 ctypes.POINTER(KdaActivation), _VP, _VP, _VP, _SZ, _VP, _VP]),
    "kda_chunk_bwd_act": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape),
                                ctypes.POINTER(KdaActivation), _VP, _VP, _VP, _VP, _VP, _VP,
                                _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "kda_chunk_fwd_noalloc": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape),
                                    _VP, _VP, _VP, _VP]),
    "kda_recurrent_fwd": (_ST, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(KdaShape),
                                _VP, _VP, _VP, _VP]),
    "kda_read_device_status": (_ST, [_VP, ctypes.POINTER(ctypes.c_int32), _VP]),
    "kda_clear_device_status": (_ST, [_VP, _VP]),
    "kda_status_string": (ctypes.c_char_p, [_ST]),
    "kda_last_error_message": (ctypes.c_char_p, []),
    "kda_version": (ctypes.c_char_p, []),
    "kda_profile_enable": (_ST, [ctypes.c_int]),
    "kda_profile_report": (ctypes.c_int, [ctypes.c_char_p, _SZ, ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_int64), ctypes.c_int]),
    "kda_profile_reset": (None, []),
    "kda_measure_fp32_fma_peak": (_ST, [ctypes.POINTER(ctypes.c_double), _VP]),
}


def load() -> ctypes.CDLL:
    """Load libkda_gb300.so (built by `gated_delta_rule_cumsum_gb300.build.build()`)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {_LIB_PATH} is missing "
                "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _LIB = lib
    return _LIB


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> Optional[ctypes.c_void_p]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int):
    if status != KDA_OK:
        raise KdaError(status, load().kda_last_error_message().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_DTYPE_BF16
    if t.dtype == torch.float32:
        return KDA_DTYPE_F32
    raise KdaError(KDA_ERR_UNSUPPORTED, f"dtype {t.dtype} (supported: bfloat16, float32)")


def make_shape(q: torch.Tensor, v: torch.Tensor, cu_seqlens: Optional[torch.Tensor] = None,
               scale: Optional[float] = None, g_scale: float = 1.0, flags: int = 0) -> KdaShape:
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    return KdaShape(B, T, H, HV, K, V, N, _dtype_code(q), -1.0 if scale is None else float(scale),
                    float(g_scale), int(flags))


# ------------------------------------------------------------------ the C calls
def kda_gate_cumsum(g, g_cum, cu_seqlens, shape: KdaShape, chunk_size: int, dev_status=None,
                    stream=None):
    _check(load().kda_gate_cumsum(_ptr(g), _ptr(g_cum), _ptr(cu_seqlens), ctypes.byref(shape),
                                  int(chunk_size), _ptr(dev_status), _stream(stream)))


def kda_gate_cumsum_act(g, g_cum, cu_seqlens, shape: KdaShape, act: KdaActivation,
                        chunk_size: int, dev_status=None, stream=None):
    _check(load().kda_gate_cumsum_act(_ptr(g), _ptr(g_cum), _ptr(cu_seqlens), ctypes.byref(shape),
                                      ctypes.byref(act), int(chunk_size), _ptr(dev_status),
                                      _stream(stream)))


def kda_chunk_fwd_act(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, act: KdaActivation, o,
                      ht, workspace, dev_status=None, stream=None):
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kda_chunk_fwd_act(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(cu_seqlens), ctypes.byref(shape), ctypes.byref(act),
                                    _ptr(o), _ptr(ht), _ptr(workspace), nbytes, _ptr(dev_status),
                                    _stream(stream)))


def kda_recurrent_fwd_act(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, act: KdaActivation,
                          o, ht, dev_status=None, stream=None):
    _check(load().kda_recurrent_fwd_act(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                        _ptr(cu_seqlens), ctypes.byref(shape), ctypes.byref(act),
                                        _ptr(o), _ptr(ht), _ptr(dev_status), _stream(stream)))


def kda_chunk_fwd(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, o, ht, workspace,
                  dev_status=None, stream=None):
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                _ptr(cu_seqlens), ctypes.byref(shape), _ptr(o), _ptr(ht),
                                _ptr(workspace), nbytes, _ptr(dev_status), _stream(stream)))


def kda_chunk_fwd_noalloc(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, o, ht,
                          dev_status=None, stream=None):
    """kda_chunk_fwd without a workspace: the library's built-in scratch array
    (KDA_NOALLOC_SCRATCH_BYTES) stands in for it; calls must not overlap."""
    _check(load().kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        _ptr(h0), _ptr(cu_seqlens), ctypes.byref(shape), _ptr(o),
                                        _ptr(ht), _ptr(dev_status), _stream(stream)))


KDA_NOALLOC_SCRATCH_BYTES = 32 << 20


def kda_chunk_workspace_size(shape: KdaShape) -> int:
    return int(load().kda_chunk_workspace_size(ctypes.byref(shape)))


def kda_workspace_size(shape: KdaShape) -> int:
    """kda_chunk_workspace_size under the boundary's original name."""
    return int(load().kda_workspace_size(ctypes.byref(shape)))


def kda_recurrent_bwd_workspace_size(shape: KdaShape) -> int:
    return int(load().kda_recurrent_bwd_workspace_size(ctypes.byref(shape)))


def kda_recurrent_bwd(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, dout, dht, dq, dk, dv,
                      dg, dbeta, dh0, workspace, dev_status=None, stream=None):
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kda_recurrent_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(cu_seqlens), ctypes.byref(shape), _ptr(dout), _ptr(dht),
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
                                    _ptr(dh0), _ptr(workspace), ws, _ptr(dev_status),
                                    _stream(stream)))


def kda_chunk_bwd_workspace_size(shape: KdaShape) -> int:
    return int(load().kda_chunk_bwd_workspace_size(ctypes.byref(shape)))


def kda_chunk_bwd(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, dout, dht, dq, dk, dv, dg,
                  dbeta, dh0, workspace, dev_status=None, stream=None):
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kda_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                _ptr(cu_seqlens), ctypes.byref(shape), _ptr(dout), _ptr(dht),
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0),
                                _ptr(workspace), ws, _ptr(dev_status), _stream(stream)))


def kda_chunk_fwd_save(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, act, o, ht, workspace,
                       dev_status=None, stream=None):
    """`act`: a KdaActivation or None."""
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kda_chunk_fwd_save(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                     _ptr(cu_seqlens), ctypes.byref(shape),
                                     None if act is None else ctypes.byref(act), _ptr(o), _ptr(ht),
                                     _ptr(workspace), ws, _ptr(dev_status), _stream(stream)))


def kda_chunk_bwd_act(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, act: KdaActivation,
                      dout, dht, dq, dk, dv, dg, dbeta, dh0, dA_log, ddt_bias, workspace,
                      dev_status=None, stream=None):
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kda_chunk_bwd_act(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(cu_seqlens), ctypes.byref(shape), ctypes.byref(act),
                                    _ptr(dout), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                                    _ptr(dg), _ptr(dbeta), _ptr(dh0), _ptr(dA_log),
                                    _ptr(ddt_bias), _ptr(workspace), ws, _ptr(dev_status),
                                    _stream(stream)))


def kda_recurrent_bwd_act(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, act: KdaActivation,
                          dout, dht, dq, dk, dv, dg, dbeta, dh0, dA_log, ddt_bias, workspace,
                          dev_status=None, stream=None):
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().kda_recurrent_bwd_act(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                        _ptr(cu_seqlens), ctypes.byref(shape), ctypes.byref(act),
                                        _ptr(dout), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                                        _ptr(dg), _ptr(dbeta), _ptr(dh0), _ptr(dA_log),
                                        _ptr(ddt_bias), _ptr(workspace), ws, _ptr(dev_status),
                                        _stream(stream)))


def kda_recurrent_fwd(q, k, v, g, beta, h0, cu_seqlens, shape: KdaShape, o, ht, dev_status=None,
                      stream=None):
    _check(load().kda_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(cu_seqlens), ctypes.byref(shape), _ptr(o), _ptr(ht),
                                    _ptr(dev_status), _stream(stream)))


def kda_read_device_status(dev_status, stream=None):
    """Synchronises the stream; returns (status, bits)."""
    bits = ctypes.c_int32(0)
    st = load().kda_read_device_status(_ptr(dev_status), ctypes.byref(bits), _stream(stream))
    return int(st), int(bits.value)


def kda_clear_device_status(dev_status, stream=None):
    _check(load().kda_clear_device_status(_ptr(dev_status), _stream(stream)))


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def kda_last_error_message() -> str:
    return load().kda_last_error_message().decode()


def kda_version() -> str:
    return load().kda_version().decode()


def kda_profile_enable(enable: bool = True):
    _check(load().kda_profile_enable(int(bool(enable))))


def kda_profile_reset():
    load().kda_profile_reset()


def kda_measure_fp32_fma_peak(stream=None) -> float:
    """The device's fp32 FMA peak in TFLOP/s, measured by an FMA-loop kernel."""
    out = ctypes.c_double(0.0)
    _check(load().kda_measure_fp32_fma_peak(ctypes.byref(out), _stream(stream)))
    return float(out.value)


def kda_profile_report(max_entries: int = 32) -> dict:
    """{kernel name: (total ms, launches)} of the kernels timed since the last reset."""
    names = ctypes.create_string_buffer(4096)
    ms = (ctypes.c_double * max_entries)()
    cnt = (ctypes.c_int64 * max_entries)()
    n = load().kda_profile_report(names, len(names), ms, cnt, max_entries)
    if n < 0:
        raise KdaError(KDA_ERR_CUDA, "kda_profile_report failed")
    labels = names.raw.split(b"\0")[:n]
    return {labels[i].decode(): (ms[i], int(cnt[i])) for i in range(n)}


# ------------------------------------------------------- allocating wrappers
def _one_device(*ts):
    """Every given tensor on the same CUDA device, else KdaError (pointers of
    another device, or of the host, must never reach the kernels)."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise KdaError(KDA_ERR_INVALID_ARG, "tensors must be on a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise KdaError(KDA_ERR_INVALID_ARG,
                           f"tensors must be on one CUDA device ({dev} and {t.device})")
    return dev


def _on_tensor_device(fn):
    """Run fn with its first CUDA tensor's device as the current device: the library
    launches on the current device and takes that device's current stream."""
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        for x in itertools.chain(args, kwargs.values()):
            if isinstance(x, torch.Tensor) and x.is_cuda:
                with torch.cuda.device(x.device):
                    return fn(*args, **kwargs)
        return fn(*args, **kwargs)
    return wrapper


def _prep(*ts):
    for t in ts:
        if t is not None and t.requires_grad:
            raise KdaError(KDA_ERR_UNSUPPORTED,
                           "inputs requiring grad are rejected here: use kda_autograd")
    _one_device(*ts)
    return [None if t is None else t.contiguous() for t in ts]


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


@_on_tensor_device
def gate_cumsum(g, cu_seqlens=None, chunk_size: int = 64, g_scale: float = 1.0, dev_status=None,
                stream=None, A_log=None, dt_bias=None):
    """Chunk-local cumsum of g [B,T,HV,K] fp32; rows outside every sequence are zero.
    With `A_log`, g is the raw gate, activated first (see chunk_kda)."""
    g, cu_seqlens = _prep(g, cu_seqlens)
    _one_device(g, dev_status, A_log, dt_bias)
    B, T, HV, K = g.shape
    shape = KdaShape(B, T, 1, HV, K, 1, B if cu_seqlens is None else cu_seqlens.numel() - 1,
                     KDA_DTYPE_F32, -1.0, float(g_scale), 0)
    out = torch.zeros_like(g)
    if A_log is not None:
        kda_gate_cumsum_act(g, out, cu_seqlens, shape, make_activation(A_log, dt_bias),
                            chunk_size, dev_status, stream)
    else:
        kda_gate_cumsum(g, out, cu_seqlens, shape, chunk_size, dev_status, stream)
    return out


@_on_tensor_device
def chunk_kda(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
              cu_seqlens=None, use_qk_l2norm_in_kernel=False, g_scale=1.0, g_is_cumsum=False,
              split_scan=False, A_log=None, dt_bias=None, beta_sigmoid_scale=0.0,
              workspace=None, dev_status=None, stream=None, serial=False):
    """Chunked forward; returns (o, ht or None).  `g` is the per-token log2 gate, or
    with `A_log` the raw gate (activated inside: -exp(A_log) softplus(g + dt_bias),
    times g_scale); `beta_sigmoid_scale` > 0 makes `beta` logits."""
    q, k, v, g, beta, h0, cu = _prep(q, k, v, g, beta, initial_state, cu_seqlens)
    _one_device(q, workspace, dev_status, A_log, dt_bias)
    flags = (KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0) | (
        KDA_FLAG_G_IS_CUMSUM if g_is_cumsum else 0) | (KDA_FLAG_SPLIT_SCAN if split_scan else 0) | (
        KDA_FLAG_SERIAL if serial else 0)
    shape = make_shape(q, v, cu, scale, g_scale, flags)
    o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    ht = (torch.empty(shape.num_seqs, shape.HV, shape.K, shape.V, dtype=torch.float32,
                      device=q.device) if output_final_state else None)
    if workspace is None:
        workspace = torch.empty(max(kda_chunk_workspace_size(shape), 256), dtype=torch.uint8,
                                device=q.device)
    if A_log is not None or beta_sigmoid_scale:
        act = make_activation(A_log, dt_bias, beta_sigmoid_scale)
        kda_chunk_fwd_act(q, k, v, g, beta, h0, cu, shape, act, o, ht, workspace, dev_status,
                          stream)
    else:
        kda_chunk_fwd(q, k, v, g, beta, h0, cu, shape, o, ht, workspace, dev_status, stream)
    return o, ht


@_on_tensor_device
def recurrent_kda_backward(q, k, v, gate, beta, dout, initial_state=None, dht=None, *,
                           cu_seqlens=None, scale=None, g_scale=1.0, want_dh0=True,
                           use_qk_l2norm_in_kernel=False, A_log=None, dt_bias=None,
                           beta_sigmoid_scale=0.0, dev_status=None, stream=None):
    """Gradients of the token recurrence for an output gradient `dout` and a final-state
    gradient `dht` (or None): a dict of fp32 tensors dq, dk, dv, dg (with respect to the
    per-token log2 gate), dbeta and dh0 (None unless `want_dh0`).  With `A_log` (and
    `dt_bias`, `beta_sigmoid_scale`) the inputs are raw as in chunk_kda: dg and dbeta are
    the raw inputs' gradients and the dict adds dA_log and ddt_bias."""
    ts = [q, k, v, gate, beta, dout, initial_state, dht, cu_seqlens, A_log, dt_bias, dev_status]
    _one_device(*ts)
    ts = ts[:-1]
    q, k, v, g, beta, dout, h0, dht, cu, A_log, dt_bias = [
        None if t is None else t.detach().contiguous() for t in ts]
    shape = make_shape(q, v, cu, scale, g_scale,
                       KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0)
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty(q.shape, **f32), dk=torch.empty(k.shape, **f32),
               dv=torch.empty(v.shape, **f32), dg=torch.empty(g.shape, **f32),
               dbeta=torch.empty(beta.shape, **f32),
               dh0=(torch.empty(shape.num_seqs, shape.HV, shape.K, shape.V, **f32)
                    if want_dh0 else None))
    ws = torch.empty(max(kda_recurrent_bwd_workspace_size(shape), 16), dtype=torch.uint8,
                     device=q.device)
    if A_log is not None or beta_sigmoid_scale:
        out["dA_log"] = None if A_log is None else torch.empty(A_log.shape, **f32)
        out["ddt_bias"] = None if dt_bias is None else torch.empty(dt_bias.shape, **f32)
        kda_recurrent_bwd_act(q, k, v, g, beta, h0, cu, shape,
                              make_activation(A_log, dt_bias, beta_sigmoid_scale), dout, dht,
                              out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"], out["dh0"],
                              out["dA_log"], out["ddt_bias"], ws, dev_status, stream)
    else:
        kda_recurrent_bwd(q, k, v, g, beta, h0, cu, shape, dout, dht, out["dq"], out["dk"],
                          out["dv"], out["dg"], out["dbeta"], out["dh0"], ws, dev_status, stream)
    return out


@_on_tensor_device
def chunk_kda_forward_save(q, k, v, g, beta, scale=None, initial_state=None,
                           output_final_state=False, cu_seqlens=None,
                           use_qk_l2norm_in_kernel=False, g_scale=1.0, A_log=None, dt_bias=None,
                           beta_sigmoid_scale=0.0, workspace=None, dev_status=None, stream=None,
                           serial=False):
    """chunk_kda (the same o and ht) by kda_chunk_fwd_save: returns (o, ht or None,
    saved), `saved` the uint8 workspace that a later chunk_kda_backward(..., saved=saved)
    of the same inputs and options reads instead of running the forward again
    (bf16 inputs, K = V = 128)."""
    q, k, v, g, beta, h0, cu = _prep(q, k, v, g, beta, initial_state, cu_seqlens)
    _one_device(q, workspace, dev_status, A_log, dt_bias)
    flags = (KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0) | (
        KDA_FLAG_SERIAL if serial else 0)
    shape = make_shape(q, v, cu, scale, g_scale, flags)
    o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    ht = (torch.empty(shape.num_seqs, shape.HV, shape.K, shape.V, dtype=torch.float32,
                      device=q.device) if output_final_state else None)
    if workspace is None:
        workspace = torch.empty(max(kda_chunk_bwd_workspace_size(shape), 256), dtype=torch.uint8,
                                device=q.device)
    act = (make_activation(A_log, dt_bias, beta_sigmoid_scale)
           if A_log is not None or beta_sigmoid_scale else None)
    kda_chunk_fwd_save(q, k, v, g, beta, h0, cu, shape, act, o, ht, workspace, dev_status, stream)
    return o, ht, workspace


@_on_tensor_device
def chunk_kda_backward(q, k, v, gate, beta, dout, initial_state=None, dht=None, *,
                       cu_seqlens=None, scale=None, g_scale=1.0, want_dh0=True,
                       use_qk_l2norm_in_kernel=False, A_log=None, dt_bias=None,
                       beta_sigmoid_scale=0.0, dev_status=None, stream=None, workspace=None,
                       saved=None):
    """The gradients recurrent_kda_backward returns (dq, dk, dv, dg, dbeta, dh0 as fp32,
    and with the activations dA_log and ddt_bias), computed by kda_chunk_bwd in the
    chunked form on the tensor cores (bf16 inputs, K = V = 128).  `workspace`, if
    given, is a uint8 device tensor of at least kda_chunk_bwd_workspace_size bytes;
    `saved`, chunk_kda_forward_save's workspace for the same inputs and options: the
    backward then starts from what it holds (KDA_FLAG_BWD_SAVED)."""
    if saved is not None:
        workspace = saved
    ts = [q, k, v, gate, beta, dout, initial_state, dht, cu_seqlens, A_log, dt_bias, dev_status,
          workspace]
    _one_device(*ts)
    q, k, v, g, beta, dout, h0, dht, cu, A_log, dt_bias = [
        None if t is None else t.detach().contiguous() for t in ts[:11]]
    shape = make_shape(q, v, cu, scale, g_scale,
                       (KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0) |
                       (KDA_FLAG_BWD_SAVED if saved is not None else 0))
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty(q.shape, **f32), dk=torch.empty(k.shape, **f32),
               dv=torch.empty(v.shape, **f32), dg=torch.empty(g.shape, **f32),
               dbeta=torch.empty(beta.shape, **f32),
               dh0=(torch.empty(shape.num_seqs, shape.HV, shape.K, shape.V, **f32)
                    if want_dh0 else None))
    if workspace is None:
        workspace = torch.empty(max(kda_chunk_bwd_workspace_size(shape), 256), dtype=torch.uint8,
                                device=q.device)
    if A_log is not None or beta_sigmoid_scale:
        out["dA_log"] = None if A_log is None else torch.empty(A_log.shape, **f32)
        out["ddt_bias"] = None if dt_bias is None else torch.empty(dt_bias.shape, **f32)
        kda_chunk_bwd_act(q, k, v, g, beta, h0, cu, shape,
                          make_activation(A_log, dt_bias, beta_sigmoid_scale), dout, dht,
                          out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"], out["dh0"],
                          out["dA_log"], out["ddt_bias"], workspace, dev_status, stream)
    else:
        kda_chunk_bwd(q, k, v, g, beta, h0, cu, shape, dout, dht, out["dq"], out["dk"],
                      out["dv"], out["dg"], out["dbeta"], out["dh0"], workspace, dev_status,
                      stream)
    return out


class _KdaFunction(torch.autograd.Function):
    """Forward by the chunked (or token) kernels, backward by kda_chunk_bwd or
    kda_recurrent_bwd: the chunked form computes the recurrence, so its gradients
    are the recurrence's."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, h0, cu, scale, g_scale, chunked, l2norm, A_log, dt_bias,
                beta_sigmoid_scale, save):
        ctx.saved = None
        with torch.no_grad():
            kw = dict(cu_seqlens=cu, output_final_state=True, scale=scale, g_scale=g_scale,
                      use_qk_l2norm_in_kernel=l2norm,
                      A_log=None if A_log is None else A_log.detach(),
                      dt_bias=None if dt_bias is None else dt_bias.detach(),
                      beta_sigmoid_scale=beta_sigmoid_scale)
            if chunked and save and _chunk_bwd_applies(q, v):
                # the forward that keeps what the chunked backward would recompute
                o, ht, ctx.saved = chunk_kda_forward_save(
                    q.detach(), k.detach(), v.detach(), g.detach(), beta.detach(),
                    initial_state=None if h0 is None else h0.detach(), **kw)
            elif chunked:
                o, ht = chunk_kda(q.detach(), k.detach(), v.detach(), g.detach(), beta.detach(),
                                  initial_state=None if h0 is None else h0.detach(), **kw)
            else:
                o, ht = recurrent_kda(q.detach(), k.detach(), v.detach(), g.detach(),
                                      beta.detach(),
                                      None if h0 is None else h0.detach(), **kw)
        ctx.save_for_backward(q, k, v, g, beta, h0, cu, A_log, dt_bias)
        ctx.scale, ctx.g_scale, ctx.l2norm = scale, g_scale, l2norm
        ctx.beta_sigmoid_scale = beta_sigmoid_scale
        return o, ht

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g, beta, h0, cu, A_log, dt_bias = ctx.saved_tensors
        # kda_recurrent_bwd takes dL/do in the inputs' dtype: with bf16 inputs the
        # upstream gradient is rounded to bf16 here (a relative change of at most
        # 2^-9 per element) before the fp32 backward uses it.
        do = torch.zeros_like(v) if do is None else do.to(q.dtype)
        gr = None
        if _chunk_bwd_applies(q, v):
            # the chunked backward on the tensor cores; a chunk whose gate range it
            # does not take is reported on the status word, and then the token
            # recurrence's backward runs instead (this reads the word: one sync)
            st = new_status(q.device)
            gr = chunk_kda_backward(q, k, v, g, beta, do, h0, dht, cu_seqlens=cu,
                                    scale=ctx.scale, g_scale=ctx.g_scale,
                                    want_dh0=h0 is not None, use_qk_l2norm_in_kernel=ctx.l2norm,
                                    A_log=A_log, dt_bias=dt_bias,
                                    beta_sigmoid_scale=ctx.beta_sigmoid_scale, dev_status=st,
                                    saved=ctx.saved)
            ctx.saved = None
            if kda_read_device_status(st)[1] & KDA_DEVICE_GATE_RANGE:
                gr = None
        if gr is None:
            gr = recurrent_kda_backward(q, k, v, g, beta, do, h0, dht, cu_seqlens=cu,
                                        scale=ctx.scale, g_scale=ctx.g_scale,
                                        want_dh0=h0 is not None,
                                        use_qk_l2norm_in_kernel=ctx.l2norm, A_log=A_log,
                                        dt_bias=dt_bias, beta_sigmoid_scale=ctx.beta_sigmoid_scale)
        dh0 = gr["dh0"] if h0 is not None else None
        dA = None if A_log is None else gr["dA_log"].to(A_log.dtype)
        ddt = None if dt_bias is None else gr["ddt_bias"].to(dt_bias.dtype)
        return (gr["dq"].to(q.dtype), gr["dk"].to(k.dtype), gr["dv"].to(v.dtype),
                gr["dg"].to(g.dtype), gr["dbeta"].to(beta.dtype), dh0, None, None, None, None,
                None, dA, ddt, None, None)


@_on_tensor_device
def _chunk_bwd_applies(q, v):
    return q.dtype == torch.bfloat16 and q.shape[3] == 128 and v.shape[3] == 128


def kda_autograd(q, k, v, g, beta, initial_state=None, *, cu_seqlens=None, scale=None,
                 g_scale=1.0, chunked=True, use_qk_l2norm_in_kernel=False, A_log=None,
                 dt_bias=None, beta_sigmoid_scale=0.0, save_for_backward=True):
    """(o, ht) with gradients: forward by chunk_kda (or recurrent_kda when `chunked` is
    False), backward by kda_chunk_bwd where it applies (bf16, K = V = 128), else
    kda_recurrent_bwd; `g` is the per-token log2 gate,
    or with `A_log` the raw gate (A_log and dt_bias then receive gradients too).
    With `save_for_backward` (and the chunked backward applying) the forward keeps
    the backward's recomputed state (kda_chunk_fwd_save: kda_chunk_bwd_workspace_size
    bytes held until the backward) and the backward does not run the forward again;
    False recomputes it in the backward."""
    _one_device(q, k, v, g, beta, initial_state, cu_seqlens, A_log, dt_bias)
    return _KdaFunction.apply(q, k, v, g, beta, initial_state, cu_seqlens, scale, g_scale, chunked,
                              bool(use_qk_l2norm_in_kernel), A_log, dt_bias,
                              float(beta_sigmoid_scale), bool(save_for_backward))


@_on_tensor_device
def recurrent_kda(q, k, v, gate, beta, initial_state=None, *, cu_seqlens=None,
                  output_final_state=False, scale=None, use_qk_l2norm_in_kernel=False,
                  g_scale=1.0, A_log=None, dt_bias=None, beta_sigmoid_scale=0.0,
                  dev_status=None, stream=None, final_state_out=None):
    """Token-by-token forward; returns (o, ht or None).  `gate` is the per-token log2 gate
    (or, with `A_log`, the raw gate; see chunk_kda)."""
    q, k, v, g, beta, h0, cu = _prep(q, k, v, gate, beta, initial_state, cu_seqlens)
    _one_device(q, dev_status, final_state_out, A_log, dt_bias)
    flags = KDA_FLAG_QK_L2NORM if use_qk_l2norm_in_kernel else 0
    shape = make_shape(q, v, cu, scale, g_scale, flags)
    o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    ht = final_state_out
    if ht is None and output_final_state:
        ht = torch.empty(shape.num_seqs, shape.HV, shape.K, shape.V, dtype=torch.float32,
                         device=q.device)
    if A_log is not None or beta_sigmoid_scale:
        act = make_activation(A_log, dt_bias, beta_sigmoid_scale)
        kda_recurrent_fwd_act(q, k, v, g, beta, h0, cu, shape, act, o, ht, dev_status, stream)
    else:
        kda_recurrent_fwd(q, k, v, g, beta, h0, cu, shape, o, ht, dev_status, stream)
    return o, ht
