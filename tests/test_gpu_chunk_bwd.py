"""kda_chunk_bwd (the chunked backward on the tensor cores) against the fp64 oracle's
gradients, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

from oracle import chunk_backward as ocb
from tests import parity
from tests.test_gpu_recurrent import _packed, _small
from tests.test_gpu_recurrent_bwd import _grads_in, _np

pytestmark = pytest.mark.gpu

# max |error| / max |gradient| per gradient.  The operands of every product are bf16
# (the inputs, the state and v' checkpoints, the intermediate gradients dv', dh,
# dw, dAkk, dP, dA) with fp32 accumulation: a few bf16 roundings (2^-9 = 2e-3 each)
# in a chain, and dg sums them over up to 64 rows.  Measured: at most 4.7e-3.
TOL = 1e-2
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def _oracle(inp, dout, dht, g_scale=1.0, heads=None):
    """chunk_grads on the value heads `heads` (with their q/k heads; all by default)."""
    q, k, v, g, beta, h0 = (inp[x] for x in ("q", "k", "v", "g", "beta", "h0"))
    cu = inp["cu_seqlens"]
    if heads is not None:
        grp = v.shape[2] // q.shape[2]
        assert grp == 1
        q, k, v, g, beta = (t[:, :, heads] for t in (q, k, v, g, beta))
        dout = dout[:, :, heads]
        h0 = None if h0 is None else h0[:, heads]
        dht = None if dht is None else dht[:, heads]
    return ocb.chunk_grads(_np(q), _np(k), _np(v), _np(g), _np(beta), _np(dout), _np(h0),
                           _np(dht), cu_seqlens=None if cu is None else cu.cpu().numpy(),
                           g_scale=g_scale)


def _run(kda, inp, dout, dht, **kw):
    return kda.chunk_kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout,
                                  inp["h0"], dht, cu_seqlens=inp["cu_seqlens"], **kw)


def _errors(got, ref, rows=None, heads=None):
    errs = {}
    for name in NAMES:
        if ref.get(name) is None or got.get(name) is None:
            continue
        g = got[name]
        if heads is not None:
            g = g[:, heads] if name == "dh0" else g[:, :, heads]
        g, r = _np(g), ref[name]
        if rows is not None and name != "dh0":
            g, r = g[:, :rows], r[:, :rows]
        errs[name] = parity.rel_err(g, r)
    return errs


def _check(got, ref, **kw):
    errs = _errors(got, ref, **kw)
    print(errs)
    bad = {n: e for n, e in errs.items() if not e <= TOL}
    assert not bad, errs


@pytest.mark.parametrize("B,T,H,HV,h0,dht", [
    (2, 200, 2, 2, True, True),     # three full chunks and a ragged one per sequence
    (1, 64, 1, 1, False, False),    # one chunk from a zero state, no final-state gradient
    (1, 130, 1, 2, True, True),     # two value heads share each q/k row (summed dq, dk)
    (1, 700, 2, 2, True, True),     # eleven chunks
])
def test_dense(kda_lib, B, T, H, HV, h0, dht):
    inp = _small(1300 + T + HV, B=B, T=T, H=H, HV=HV, K=128, V=128, h0=h0, g_hi=0.3)
    dout, dh = _grads_in(inp, T)
    if not dht:
        dh = None
    st = kda_lib.new_status()
    got = _run(kda_lib, inp, dout, dh, dev_status=st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    _check(got, _oracle(inp, dout, dh))


def test_packed_with_empty_slots_and_nan_tail(kda_lib):
    lens = [5, 0, 64, 130, 1, 0, 77]
    inp = _packed(1361, lens, HV=2, H=2, K=128, V=128)
    dout, dht = _grads_in(inp, 1362)
    st = kda_lib.new_status()
    got = _run(kda_lib, inp, dout, dht, dev_status=st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    end = sum(lens)
    _check(got, _oracle(inp, dout, dht), rows=end)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):  # rows past the last offset stay zero
        assert torch.all(got[name][:, end:] == 0), name
    for n, L in enumerate(lens):
        if L == 0:  # an empty slot passes the state gradient through
            assert torch.equal(got["dh0"][n], dht[n])


def test_natural_log_gate_scale(kda_lib):
    inp = _small(1371, B=1, T=100, H=1, HV=1, K=128, V=128, g_hi=0.2)
    dout, dht = _grads_in(inp, 1372)
    gs = 1.0 / np.log(2.0)
    got = _run(kda_lib, inp, dout, dht, g_scale=gs)
    _check(got, _oracle(inp, dout, dht, g_scale=gs))


def test_gate_range_beyond_the_split_grams_is_reported(kda_lib):
    """A chunk whose cumulative gate falls below -100 (log2) is refused with a status bit."""
    inp = _small(1381, B=1, T=128, H=1, HV=1, K=128, V=128)
    inp["g"][:, 64:] = -3.0  # 64 rows of -3: the second chunk reaches -192
    dout, dht = _grads_in(inp, 1382)
    st = kda_lib.new_status()
    _run(kda_lib, inp, dout, dht, dev_status=st)
    status, bits = kda_lib.kda_read_device_status(st)
    assert bits & kda_lib.KDA_DEVICE_GATE_RANGE and status == kda_lib.KDA_ERR_UNSUPPORTED


def test_training_shape_sampled_heads(kda_lib):
    """B = 1, T = 8192, H = HV = 16, K = V = 128: heads 0 and 15 against the oracle."""
    import kda_synth

    inp = kda_synth.make_inputs(1, device="cuda")
    dout, dht = _grads_in(inp, 1391)
    got = _run(kda_lib, inp, dout, dht)
    heads = [0, 15]
    _check(got, _oracle(inp, dout, dht, heads=heads), heads=heads)


@pytest.mark.parametrize("wide_gate", [False, True])
def test_autograd_takes_the_chunked_backward(kda_lib, wide_gate):
    """loss.backward() through kda_autograd with bf16, K = V = 128: kda_chunk_bwd, or,
    for a chunk whose gate range it refuses, the token recurrence's backward."""
    inp = _small(1401, B=1, T=150, H=1, HV=1, K=128, V=128, g_hi=0.3)
    if wide_gate:
        inp["g"][:, 64:128] = -3.0
    dout, dht = _grads_in(inp, 1402)
    leaves = {n: inp[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "h0")}
    o, ht = kda_lib.kda_autograd(leaves["q"], leaves["k"], leaves["v"], leaves["g"],
                                 leaves["beta"], leaves["h0"])
    ((o.float() * dout.float()).sum() + (ht * dht).sum()).backward()
    ref = _oracle(inp, dout, dht)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                      ("h0", "dh0")):
        got = leaves[name].grad
        err = parity.rel_err(got, ref[key])
        assert err <= TOL, (name, err)


def test_pipelined_reverse_scan_matches_serial_and_oracle(kda_lib):
    """Two sequences of 32 chunks (the last one ragged) over 8 heads: the call pipelines
    the reverse scan with the gradient kernel (split at chunk 27 on 152 SMs), bit for bit
    the serial call's result (no atomics when HV == H), and the oracle's on two heads."""
    inp = _small(1411, B=2, T=2000, H=8, HV=8, K=128, V=128, g_hi=0.3)
    dout, dht = _grads_in(inp, 1412)
    q, k, v, g, beta, h0 = (inp[n] for n in ("q", "k", "v", "g", "beta", "h0"))
    outs = []
    for flags in (0, kda_lib.KDA_FLAG_SERIAL):
        shape = kda_lib.make_shape(q, v, None, flags=flags)
        ws = torch.empty(kda_lib.kda_chunk_bwd_workspace_size(shape), dtype=torch.uint8,
                         device="cuda")
        f32 = dict(dtype=torch.float32, device="cuda")
        gr = dict(dq=torch.empty(q.shape, **f32), dk=torch.empty(k.shape, **f32),
                  dv=torch.empty(v.shape, **f32), dg=torch.empty(g.shape, **f32),
                  dbeta=torch.empty(beta.shape, **f32), dh0=torch.empty(h0.shape, **f32))
        st = kda_lib.new_status()
        kda_lib.kda_chunk_bwd(q, k, v, g, beta, h0, None, shape, dout, dht, gr["dq"], gr["dk"],
                              gr["dv"], gr["dg"], gr["dbeta"], gr["dh0"], ws, st)
        assert kda_lib.kda_read_device_status(st) == (0, 0)
        outs.append(gr)
    for name in NAMES:
        assert torch.equal(outs[0][name], outs[1][name]), name
    heads = [0, 7]
    _check(outs[0], _oracle(inp, dout, dht, heads=heads), heads=heads)
