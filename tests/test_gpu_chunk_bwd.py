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
    the reverse scan with the gradient kernel (split at chunk 27 on 152 SMs) and the
    forward's re-run in parts (a part's first chunk forms v' from its start state rather
    than from the previous chunk's state and v', which rounds differently): within a few
    bf16 roundings of the serial call's result, and the oracle's on two heads."""
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
        err = parity.rel_err(outs[0][name], outs[1][name])
        assert err <= 2e-3, (name, err)
    heads = [0, 7]
    _check(outs[0], _oracle(inp, dout, dht, heads=heads), heads=heads)


RCP_LN2 = 1.0 / np.log(2.0)


def _raw_gate(inp, seed, tail=None):
    """Raw gate and beta logits (NaN from row `tail` on), A_log and dt_bias; the raw gate
    sits low enough that a chunk's activated gate range stays inside the split grams'."""
    gen = torch.Generator().manual_seed(seed)
    B, T, HV, K = inp["g"].shape
    g_raw = torch.randn(B, T, HV, K, generator=gen) - 4.0
    b_raw = torch.randn(B, T, HV, generator=gen)
    if tail is not None:
        g_raw[:, tail:] = float("nan")
        b_raw[:, tail:] = float("nan")
    A_log = torch.log(1.0 + 3.0 * torch.rand(HV, generator=gen))
    dt_bias = 0.5 * torch.randn(HV, K, generator=gen)
    return (g_raw.cuda(), b_raw.to(torch.bfloat16).cuda(), A_log.cuda(), dt_bias.cuda())


def _oracle_opts(inp, g, beta, dout, dht, **kw):
    cu = inp["cu_seqlens"]
    g = g if isinstance(g, np.ndarray) else _np(g)
    return ocb.chunk_grads(_np(inp["q"]), _np(inp["k"]), _np(inp["v"]), g, _np(beta),
                           _np(dout), _np(inp["h0"]), _np(dht),
                           cu_seqlens=None if cu is None else cu.cpu().numpy(), **kw)


def _gate_errors(inp, dg, dA_log, ddt_bias, g_raw, A_log, dt_bias, dout, dht, end, b_raw=None,
                 **kw):
    """Errors of the raw gate's gradients, each on the scale the core's bound carries to it.

    The raw gate's gradient is the core gate's (dga) times -exp(A_log) sigmoid(g + dt_bias),
    a factor that spans two orders of magnitude here: it reweights the rows, so the
    core's bound is checked on dga, recovered by dividing the factor out.  dA_log and
    dt_bias's gradient are sums over tokens of dga times ga and times the factor; those
    sums cancel, so their errors are taken relative to the bound TOL max|dga| carried
    through the sums (error / that bound, TOL when at the bound); that bound is loose, so
    the sums are also checked as sums: the op's dA_log and dt_bias's gradient against the
    same sums over its own dga and raw-gate gradient ("_sum", fp32 reductions: 1e-5; measured below 1e-6)."""
    x = _np(g_raw)[:, :end] + _np(dt_bias)[None, None]
    a = np.exp(_np(A_log))[None, None, :, None]
    fac = -a * 0.5 * (1.0 + np.tanh(0.5 * x))
    ga = np.zeros(_np(g_raw).shape)
    ga[:, :end] = -a * np.logaddexp(0.0, x)
    core = _oracle_opts(inp, ga, inp["beta"] if b_raw is None else b_raw, dout, dht,
                        g_scale=RCP_LN2, l2norm=True, **kw)
    dga = core["dg"][:, :end]
    dmax = np.abs(dga).max()
    ref_dA = np.sum(dga * ga[:, :end], axis=(0, 1, 3))
    ref_ddt = np.sum(dga * fac, axis=(0, 1))
    got_dga = _np(dg)[:, :end] / fac
    return {"dg_core": parity.rel_err(got_dga, dga),
            "dA_log_sum": parity.rel_err(_np(dA_log),
                                         np.sum(got_dga * ga[:, :end], axis=(0, 1, 3))),
            "ddt_bias_sum": parity.rel_err(_np(ddt_bias), np.sum(_np(dg)[:, :end], axis=(0, 1))),
            "dA_log": TOL * float((np.abs(_np(dA_log) - ref_dA)
                                   / (dmax * np.abs(ga).sum(axis=(0, 1, 3)))).max()),
            "ddt_bias": TOL * float((np.abs(_np(ddt_bias) - ref_ddt)
                                     / (dmax * np.abs(fac).sum(axis=(0, 1)))).max())}


@pytest.mark.parametrize("H,HV", [(2, 2), (1, 2)])
def test_qk_l2norm_option(kda_lib, H, HV):
    """Rows of norm 3 (q) and 0.5 (k) normalised inside the op: the raw rows' gradients
    (with HV > H the normalised rows' gradients are summed before the norm's chain rule)."""
    inp = _small(1421 + HV, B=2, T=150, H=H, HV=HV, K=128, V=128, g_hi=0.3)
    inp["q"] = (inp["q"].float() * 3.0).to(torch.bfloat16)
    inp["k"] = (inp["k"].float() * 0.5).to(torch.bfloat16)
    dout, dht = _grads_in(inp, 1422)
    got = _run(kda_lib, inp, dout, dht, use_qk_l2norm_in_kernel=True)
    _check(got, _oracle_opts(inp, inp["g"], inp["beta"], dout, dht, l2norm=True))


def test_input_activations_and_l2norm_packed(kda_lib):
    """Raw gate through -exp(A_log) softplus(g + dt_bias), beta logits through the sigmoid
    and the q/k norm, packed with an empty slot and a NaN tail: the raw inputs' gradients,
    dA_log and dt_bias's."""
    lens = [70, 0, 130, 9]
    inp = _packed(1431, lens, HV=2, H=2, K=128, V=128)
    end = sum(lens)
    g_raw, b_raw, A_log, dt_bias = _raw_gate(inp, 1432, tail=end)
    dout, dht = _grads_in(inp, 1433)
    st = kda_lib.new_status()
    got = kda_lib.chunk_kda_backward(inp["q"], inp["k"], inp["v"], g_raw, b_raw, dout, inp["h0"],
                                     dht, cu_seqlens=inp["cu_seqlens"], g_scale=RCP_LN2,
                                     use_qk_l2norm_in_kernel=True, A_log=A_log, dt_bias=dt_bias,
                                     beta_sigmoid_scale=1.0, dev_status=st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    ref = _oracle_opts(inp, g_raw, b_raw, dout, dht, g_scale=RCP_LN2, l2norm=True,
                       A_log=_np(A_log), dt_bias=_np(dt_bias), beta_scale=1.0, beta_bf16=True)
    errs = _errors(got, ref, rows=end)
    errs.update(_gate_errors(inp, got["dg"], got["dA_log"], got["ddt_bias"], g_raw, A_log,
                             dt_bias, dout, dht, end, b_raw=b_raw, beta_scale=1.0,
                             beta_bf16=True))
    print(errs)
    bad = {n: e for n, e in errs.items()
           if n != "dg" and not e <= (1e-5 if n.endswith("_sum") else TOL)}
    assert not bad, errs
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.all(got[name][:, end:] == 0), name


def test_autograd_with_options_takes_the_chunked_backward(kda_lib):
    """loss.backward() through kda_autograd with the q/k norm and the gate activation."""
    inp = _small(1441, B=1, T=140, H=1, HV=1, K=128, V=128)
    g_raw, _, A_log, dt_bias = _raw_gate(inp, 1442)
    dout, dht = _grads_in(inp, 1443)
    leaves = {n: t.clone().requires_grad_(True)
              for n, t in (("q", inp["q"]), ("k", inp["k"]), ("v", inp["v"]), ("g", g_raw),
                           ("beta", inp["beta"]), ("h0", inp["h0"]), ("A_log", A_log),
                           ("dt_bias", dt_bias))}
    o, ht = kda_lib.kda_autograd(leaves["q"], leaves["k"], leaves["v"], leaves["g"],
                                 leaves["beta"], leaves["h0"], g_scale=RCP_LN2,
                                 use_qk_l2norm_in_kernel=True, A_log=leaves["A_log"],
                                 dt_bias=leaves["dt_bias"])
    ((o.float() * dout.float()).sum() + (ht * dht).sum()).backward()
    ref = _oracle_opts(inp, g_raw, inp["beta"], dout, dht, g_scale=RCP_LN2, l2norm=True,
                       A_log=_np(A_log), dt_bias=_np(dt_bias))
    errs = {key: parity.rel_err(leaves[name].grad, ref[key])
            for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"),
                              ("h0", "dh0"))}
    errs.update(_gate_errors(inp, leaves["g"].grad, leaves["A_log"].grad,
                             leaves["dt_bias"].grad, g_raw, A_log, dt_bias, dout, dht,
                             inp["q"].shape[1]))
    print(errs)
    bad = {n: e for n, e in errs.items() if not e <= (1e-5 if n.endswith("_sum") else TOL)}
    assert not bad, errs


def _save_fwd(kda, inp, **kw):
    return kda.chunk_kda_forward_save(inp["q"], inp["k"], inp["v"], kw.pop("g", inp["g"]),
                                      kw.pop("beta", inp["beta"]), initial_state=inp["h0"],
                                      output_final_state=True, cu_seqlens=inp["cu_seqlens"], **kw)


@pytest.mark.parametrize("packed", [False, True])
def test_forward_save_matches_the_forward_bitwise(kda_lib, packed):
    """kda_chunk_fwd_save returns kda_chunk_fwd's o and ht bit for bit (the backward's
    stores change no arithmetic), dense (pipelined) and packed."""
    if packed:
        inp = _packed(1451, [70, 0, 1300, 9], HV=4, H=2, K=128, V=128)
    else:
        inp = _small(1451, B=1, T=4100, H=4, HV=4, K=128, V=128)
    o, ht = kda_lib.chunk_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              initial_state=inp["h0"], output_final_state=True,
                              cu_seqlens=inp["cu_seqlens"])
    o2, ht2, _ = _save_fwd(kda_lib, inp)
    end = o.shape[1] if inp["cu_seqlens"] is None else int(inp["cu_seqlens"][-1])
    assert torch.equal(o[:, :end], o2[:, :end]) and torch.equal(ht, ht2)


@pytest.mark.parametrize("case", ["dense", "packed", "options"])
def test_saved_backward_matches_the_recomputing_one_bitwise(kda_lib, case):
    """chunk_kda_backward from chunk_kda_forward_save's workspace (KDA_FLAG_BWD_SAVED,
    no recompute) gives the recomputing call's gradients bit for bit (HV == H: no
    atomics), and the oracle's; dA_log and dt_bias's gradient are sums over tokens by
    fp32 atomics, equal to rounding."""
    kw = {}
    if case == "packed":
        inp = _packed(1461, [70, 0, 1300, 9], HV=2, H=2, K=128, V=128)
    else:
        inp = _small(1461, B=2, T=2100, H=4, HV=4, K=128, V=128, g_hi=0.3)
    dout, dht = _grads_in(inp, 1462)
    if case == "options":
        g_raw, b_raw, A_log, dt_bias = _raw_gate(inp, 1463)
        kw = dict(g=g_raw, beta=b_raw, g_scale=RCP_LN2, use_qk_l2norm_in_kernel=True,
                  A_log=A_log, dt_bias=dt_bias, beta_sigmoid_scale=1.0)
    g = kw.get("g", inp["g"])
    beta = kw.get("beta", inp["beta"])
    bkw = {n: kw[n] for n in kw if n not in ("g", "beta")}
    ref = kda_lib.chunk_kda_backward(inp["q"], inp["k"], inp["v"], g, beta, dout, inp["h0"], dht,
                                     cu_seqlens=inp["cu_seqlens"], **bkw)
    _, _, saved = _save_fwd(kda_lib, inp, **dict(kw))
    st = kda_lib.new_status()
    got = kda_lib.chunk_kda_backward(inp["q"], inp["k"], inp["v"], g, beta, dout, None, dht,
                                     cu_seqlens=inp["cu_seqlens"], saved=saved, dev_status=st,
                                     want_dh0=True, **bkw)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    for name, t in ref.items():
        if t is None:
            continue
        if name in ("dA_log", "ddt_bias"):
            assert parity.rel_err(got[name], t) <= 1e-5, name
        else:
            assert torch.equal(t, got[name]), name
    if case != "options":
        end = None if inp["cu_seqlens"] is None else int(inp["cu_seqlens"][-1])
        _check(got, _oracle(inp, dout, dht), rows=end)


def test_saved_backward_with_a_serial_call_reads_the_same_layout(kda_lib):
    """A pipelined kda_chunk_fwd_save then kda_chunk_bwd with KDA_FLAG_SERIAL |
    KDA_FLAG_BWD_SAVED through the C ABI: the workspace layout does not depend on
    KDA_FLAG_SERIAL, so the serial backward reads the pipelined forward's tiles."""
    inp = _small(1471, B=1, T=4100, H=4, HV=4, K=128, V=128, g_hi=0.3)
    dout, dht = _grads_in(inp, 1472)
    _, _, saved = _save_fwd(kda_lib, inp)
    q, k, v, g, beta = (inp[n] for n in ("q", "k", "v", "g", "beta"))
    shape = kda_lib.make_shape(q, v, None, flags=kda_lib.KDA_FLAG_SERIAL | kda_lib.KDA_FLAG_BWD_SAVED)
    f32 = dict(dtype=torch.float32, device="cuda")
    gr = dict(dq=torch.empty(q.shape, **f32), dk=torch.empty(k.shape, **f32),
              dv=torch.empty(v.shape, **f32), dg=torch.empty(g.shape, **f32),
              dbeta=torch.empty(beta.shape, **f32), dh0=torch.empty(inp["h0"].shape, **f32))
    st = kda_lib.new_status()
    kda_lib.kda_chunk_bwd(q, k, v, g, beta, None, None, shape, dout, dht, gr["dq"], gr["dk"],
                          gr["dv"], gr["dg"], gr["dbeta"], gr["dh0"], saved, st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    _check(gr, _oracle(inp, dout, dht))


def test_autograd_recomputing_backward(kda_lib):
    """kda_autograd(save_for_backward=False): the backward runs the forward again."""
    inp = _small(1481, B=1, T=150, H=1, HV=1, K=128, V=128, g_hi=0.3)
    dout, dht = _grads_in(inp, 1482)
    leaves = {n: inp[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "h0")}
    o, ht = kda_lib.kda_autograd(leaves["q"], leaves["k"], leaves["v"], leaves["g"],
                                 leaves["beta"], leaves["h0"], save_for_backward=False)
    ((o.float() * dout.float()).sum() + (ht * dht).sum()).backward()
    ref = _oracle(inp, dout, dht)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                      ("h0", "dh0")):
        err = parity.rel_err(leaves[name].grad, ref[key])
        assert err <= TOL, (name, err)


def test_saved_backward_grouped_value_heads(kda_lib):
    """Two value heads per q/k head: the saved backward's dq and dk are summed over the
    heads by atomics (order varies), so they match the recomputing call to rounding; the
    rest bit for bit."""
    inp = _small(1491, B=1, T=700, H=2, HV=4, K=128, V=128, g_hi=0.3)
    dout, dht = _grads_in(inp, 1492)
    ref = _run(kda_lib, inp, dout, dht)
    _, _, saved = _save_fwd(kda_lib, inp)
    got = kda_lib.chunk_kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout,
                                     None, dht, saved=saved, want_dh0=True)
    for name in NAMES:
        if name in ("dq", "dk"):
            assert parity.rel_err(got[name], ref[name]) <= 1e-5, name
        else:
            assert torch.equal(got[name], ref[name]), name
    _check(got, _oracle(inp, dout, dht))


def test_forward_save_refuses_the_saved_flag(kda_lib):
    """KDA_FLAG_BWD_SAVED belongs to the backward: the saving forward refuses it."""
    inp = _small(1495, B=1, T=64, H=1, HV=1, K=128, V=128)
    q, k, v, g, beta = (inp[n] for n in ("q", "k", "v", "g", "beta"))
    shape = kda_lib.make_shape(q, v, None, flags=kda_lib.KDA_FLAG_BWD_SAVED)
    ws = torch.empty(kda_lib.kda_chunk_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(v)
    with pytest.raises(kda_lib.KdaError) as err:
        kda_lib.kda_chunk_fwd_save(q, k, v, g, beta, None, None, shape, None, o, None, ws)
    assert err.value.status == kda_lib.KDA_ERR_UNSUPPORTED
