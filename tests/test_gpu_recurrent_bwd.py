"""kda_recurrent_bwd against the fp64 oracle's gradients, through the C ABI (GPU)."""
import math

import numpy as np
import pytest
import torch

from oracle import backward as ob
from tests import parity
from tests.test_gpu_recurrent import _packed, _small

pytestmark = pytest.mark.gpu

TOL = 2e-3  # max |error| / max |gradient|, per gradient (fp32 arithmetic, fp64 oracle)


def _np(t):
    return None if t is None else t.detach().float().cpu().numpy().astype(np.float64)


def _ref(inp, dout, dht, g_scale=1.0, h0_zero=False, l2norm=False):
    h0 = inp["h0"]
    if h0 is None and h0_zero:
        N, HV, K, V = inp["N"], inp["v"].shape[2], inp["q"].shape[3], inp["v"].shape[3]
        h0 = torch.zeros(N, HV, K, V)
    cu = inp["cu_seqlens"]
    return ob.recurrent_grads(_np(inp["q"]), _np(inp["k"]), _np(inp["v"]), _np(inp["g"]),
                              _np(inp["beta"]), _np(dout), _np(h0), _np(dht),
                              cu_seqlens=None if cu is None else cu.cpu().numpy(),
                              g_scale=g_scale, l2norm=l2norm)


def _run(kda, inp, dout, dht, **kw):
    return kda.recurrent_kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout,
                                      inp["h0"], dht, cu_seqlens=inp["cu_seqlens"], **kw)


def _grads_in(inp, seed):
    gen = torch.Generator().manual_seed(seed)
    dout = torch.randn(inp["v"].shape, generator=gen).to(inp["q"].dtype).cuda()
    N, HV, K, V = inp["N"], inp["v"].shape[2], inp["q"].shape[3], inp["v"].shape[3]
    dht = torch.randn(N, HV, K, V, generator=gen).cuda()
    return dout, dht


def _compare(got, ref, rows=None):
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        if ref.get(name) is None or got.get(name) is None:
            continue
        g, r = _np(got[name]), ref[name]
        if rows is not None and name != "dh0":
            g, r = g[:, :rows], r[:, :rows]
        err = parity.rel_err(g, r)
        assert err <= TOL, (name, err)


@pytest.mark.parametrize("dtype,K,V,T", [
    (torch.float32, 64, 48, 50),     # a partly used column block, ragged groups
    (torch.bfloat16, 128, 128, 40),
    (torch.float32, 32, 64, 17),     # one group plus one token
])
def test_dense(kda_lib, dtype, K, V, T):
    inp = _small(500 + K + T, B=2, T=T, H=2, HV=4, K=K, V=V, dtype=dtype)
    dout, dht = _grads_in(inp, K + V)
    got = _run(kda_lib, inp, dout, dht)
    torch.cuda.synchronize()
    _compare(got, _ref(inp, dout, dht))


def test_packed_with_empty_slots_and_nan_tail(kda_lib):
    lens = [5, 0, 17, 33, 1, 0]
    inp = _packed(61, lens, HV=4, H=2, K=64, V=48)
    dout, dht = _grads_in(inp, 62)
    st = kda_lib.new_status()
    got = _run(kda_lib, inp, dout, dht, dev_status=st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    end = sum(lens)
    _compare(got, _ref(inp, dout, dht), rows=end)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):  # rows past the last offset stay zero
        assert torch.all(got[name][:, end:] == 0), name
    for n, L in enumerate(lens):
        if L == 0:  # an empty slot passes the state gradient through bitwise
            assert torch.equal(got["dh0"][n].view(torch.int32), dht[n].view(torch.int32))


def test_natural_log_gate_scale(kda_lib):
    inp = _small(71, B=1, T=45, H=1, HV=2, K=64, V=64, dtype=torch.float32)
    dout, dht = _grads_in(inp, 72)
    got = _run(kda_lib, inp, dout, dht, g_scale=1.0 / math.log(2.0))
    _compare(got, _ref(inp, dout, dht, g_scale=1.0 / math.log(2.0)))


def test_without_initial_state_and_final_state_gradient(kda_lib):
    inp = _small(81, B=2, T=30, H=2, HV=2, K=64, V=32, h0=False, dtype=torch.float32)
    dout, _ = _grads_in(inp, 82)
    got = _run(kda_lib, inp, dout, None)
    _compare(got, _ref(inp, dout, None, h0_zero=True))


def test_grouped_value_heads_sum_into_q_and_k(kda_lib):
    inp = _small(91, B=1, T=33, H=1, HV=4, K=64, V=64, dtype=torch.float32)
    dout, dht = _grads_in(inp, 92)
    got = _run(kda_lib, inp, dout, dht)
    _compare(got, _ref(inp, dout, dht))


def test_invalid_offsets_set_the_status(kda_lib):
    """A decreasing offset: that slot is skipped with the status bit set; the others run."""
    inp = _packed(95, [10, 20, 30], HV=2, H=1, K=64, V=32)
    inp["cu_seqlens"] = torch.tensor([0, 25, 15, 60], dtype=torch.int32, device="cuda")  # decreasing
    dout, dht = _grads_in(inp, 96)
    st = kda_lib.new_status()
    got = _run(kda_lib, inp, dout, dht, dev_status=st)
    status, bits = kda_lib.kda_read_device_status(st)
    assert bits & kda_lib.KDA_DEVICE_BAD_CU_SEQLENS
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.isfinite(got[name]).all(), name


@pytest.mark.parametrize("chunked", [True, False])
def test_autograd_through_the_forward_kernels(kda_lib, chunked):
    """loss.backward() through kda_autograd: the forward kernels, then kda_recurrent_bwd;
    the gradients match the oracle's for the same dL/do and dL/dht."""
    inp = _small(97, B=1, T=70, H=2, HV=2, K=64, V=64)  # bf16: the tensor-core forward
    dout, dht = _grads_in(inp, 98)
    leaves = {n: inp[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "h0")}
    o, ht = kda_lib.kda_autograd(leaves["q"], leaves["k"], leaves["v"], leaves["g"],
                                 leaves["beta"], leaves["h0"], chunked=chunked)
    loss = (o.float() * dout.float()).sum() + (ht * dht).sum()
    loss.backward()
    ref = _ref(inp, dout, dht)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                      ("h0", "dh0")):
        got = leaves[name].grad
        # bf16 parameters receive gradients rounded to bf16
        tol = 1e-2 if got.dtype == torch.bfloat16 else TOL
        assert parity.rel_err(got, ref[key]) <= tol, (name, parity.rel_err(got, ref[key]))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_l2norm_flag(kda_lib, dtype):
    """q, k normalised inside the op: gradients of the raw rows (packed, unnormalised)."""
    inp = _packed(101, [20, 0, 37], HV=4, H=2, K=64, V=48, dtype=dtype)
    inp["q"] = (inp["q"].float() * 3.0).to(dtype)
    inp["k"] = (inp["k"].float() * 0.4).to(dtype)
    dout, dht = _grads_in(inp, 102)
    got = _run(kda_lib, inp, dout, dht, use_qk_l2norm_in_kernel=True)
    end = 57
    _compare(got, _ref(inp, dout, dht, l2norm=True), rows=end)
    assert torch.all(got["dq"][:, end:] == 0) and torch.all(got["dk"][:, end:] == 0)


def test_autograd_with_l2norm(kda_lib):
    inp = _small(103, B=1, T=50, H=2, HV=2, K=64, V=64)
    inp["q"] = (inp["q"].float() * 2.0).to(inp["q"].dtype)
    dout, dht = _grads_in(inp, 104)
    leaves = {n: inp[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "h0")}
    o, ht = kda_lib.kda_autograd(leaves["q"], leaves["k"], leaves["v"], leaves["g"],
                                 leaves["beta"], leaves["h0"], use_qk_l2norm_in_kernel=True)
    ((o.float() * dout.float()).sum() + (ht * dht).sum()).backward()
    ref = _ref(inp, dout, dht, l2norm=True)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta")):
        got = leaves[name].grad
        tol = 1e-2 if got.dtype == torch.bfloat16 else TOL
        assert parity.rel_err(got, ref[key]) <= tol, (name, parity.rel_err(got, ref[key]))


def _raw_act(inp, seed, tail=None):
    """Raw gate and beta logits for `inp` (NaN from row `tail` on), A_log, dt_bias."""
    gen = torch.Generator().manual_seed(seed)
    B, T, HV, K = inp["g"].shape
    g_raw = torch.randn(B, T, HV, K, generator=gen) - 1.5
    b_raw = torch.randn(B, T, HV, generator=gen)
    if tail is not None:
        g_raw[:, tail:] = float("nan")
        b_raw[:, tail:] = float("nan")
    A_log = torch.log(1.0 + 3.0 * torch.rand(HV, generator=gen))
    dt_bias = 0.5 * torch.randn(HV, K, generator=gen)
    return (g_raw.cuda(), b_raw.to(inp["beta"].dtype).cuda(), A_log.cuda(), dt_bias.cuda())


def _ref_act(inp, dout, dht, g_raw, b_raw, A_log, dt_bias, beta_scale):
    cu = inp["cu_seqlens"]
    return ob.recurrent_grads(_np(inp["q"]), _np(inp["k"]), _np(inp["v"]), _np(g_raw),
                              _np(b_raw), _np(dout), _np(inp["h0"]), _np(dht),
                              cu_seqlens=None if cu is None else cu.cpu().numpy(),
                              g_scale=RCP_LN2, A_log=_np(A_log), dt_bias=_np(dt_bias),
                              beta_scale=beta_scale,
                              beta_bf16=inp["beta"].dtype == torch.bfloat16)


RCP_LN2 = 1.0 / math.log(2.0)


@pytest.mark.parametrize("dtype,beta_scale", [(torch.float32, 2.0), (torch.bfloat16, 1.0)])
def test_input_activations(kda_lib, dtype, beta_scale):
    """Raw gate through -exp(A_log) softplus(g + dt_bias) and beta logits through the
    sigmoid: gradients of the raw inputs, A_log and dt_bias (packed, NaN tail)."""
    lens = [23, 0, 41, 9]
    inp = _packed(111, lens, HV=4, H=2, K=64, V=48, dtype=dtype)
    end = sum(lens)
    g_raw, b_raw, A_log, dt_bias = _raw_act(inp, 112, tail=end)
    dout, dht = _grads_in(inp, 113)
    st = kda_lib.new_status()
    got = kda_lib.recurrent_kda_backward(inp["q"], inp["k"], inp["v"], g_raw, b_raw, dout,
                                         inp["h0"], dht, cu_seqlens=inp["cu_seqlens"],
                                         g_scale=RCP_LN2, A_log=A_log, dt_bias=dt_bias,
                                         beta_sigmoid_scale=beta_scale, dev_status=st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    ref = _ref_act(inp, dout, dht, g_raw, b_raw, A_log, dt_bias, beta_scale)
    _compare(got, ref, rows=end)
    for name in ("dA_log", "ddt_bias"):
        err = parity.rel_err(_np(got[name]), ref[name])
        assert err <= TOL, (name, err)
    for name in ("dg", "dbeta"):
        assert torch.all(got[name][:, end:] == 0), name


def test_gate_activation_without_bias_or_beta_sigmoid(kda_lib):
    inp = _small(121, B=2, T=37, H=1, HV=2, K=32, V=32, dtype=torch.float32)
    g_raw, _, A_log, _ = _raw_act(inp, 122)
    dout, dht = _grads_in(inp, 123)
    got = kda_lib.recurrent_kda_backward(inp["q"], inp["k"], inp["v"], g_raw, inp["beta"], dout,
                                         inp["h0"], dht, g_scale=RCP_LN2, A_log=A_log)
    assert got["ddt_bias"] is None
    ref = _ref_act(inp, dout, dht, g_raw, inp["beta"], A_log, None, 0.0)
    _compare(got, ref)
    assert parity.rel_err(_np(got["dA_log"]), ref["dA_log"]) <= TOL


@pytest.mark.parametrize("chunked", [True, False])
def test_autograd_with_input_activations(kda_lib, chunked):
    """A_log and dt_bias as parameters: loss.backward() fills their gradients."""
    inp = _small(131, B=1, T=90, H=2, HV=2, K=64, V=64)  # bf16: the tensor-core forward
    g_raw, b_raw, A_log, dt_bias = _raw_act(inp, 132)
    dout, dht = _grads_in(inp, 133)
    leaves = {n: inp[n].clone().requires_grad_(True) for n in ("q", "k", "v", "h0")}
    leaves.update(g=g_raw.clone().requires_grad_(True), beta=b_raw.clone().requires_grad_(True),
                  A_log=A_log.clone().requires_grad_(True),
                  dt_bias=dt_bias.clone().requires_grad_(True))
    o, ht = kda_lib.kda_autograd(leaves["q"], leaves["k"], leaves["v"], leaves["g"],
                                 leaves["beta"], leaves["h0"], g_scale=RCP_LN2, chunked=chunked,
                                 A_log=leaves["A_log"], dt_bias=leaves["dt_bias"],
                                 beta_sigmoid_scale=2.0)
    ((o.float() * dout.float()).sum() + (ht * dht).sum()).backward()
    ref = _ref_act(inp, dout, dht, g_raw, b_raw, A_log, dt_bias, 2.0)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                      ("h0", "dh0"), ("A_log", "dA_log"), ("dt_bias", "ddt_bias")):
        got = leaves[name].grad
        tol = 1e-2 if got.dtype == torch.bfloat16 else TOL
        assert parity.rel_err(got, ref[key]) <= tol, (name, parity.rel_err(got, ref[key]))


def test_training_shape_directional_derivative(kda_lib):
    """At the size and in the call the benchmark times (B=1, T=8192, H=HV=16, K=V=128,
    bf16 inputs, dL/do and dL/dht drawn once): the gradients' inner product with a
    random direction d equals the central difference of L = sum(o do) + sum(ht dht)
    along d, L evaluated by the fp32 token forward on the same values.  A property
    that holds at any size, where the fp64 oracle cannot run."""
    import kda_synth

    inp = kda_synth.make_inputs(kda_synth.workload(1), device="cuda")
    names = ("q", "k", "v", "g", "beta")
    gen = torch.Generator(device="cuda").manual_seed(11)
    dout = torch.randn(inp["v"].shape, generator=gen, device="cuda").to(inp["q"].dtype)
    dht = torch.randn(1, 16, 128, 128, generator=gen, device="cuda")
    st = kda_lib.new_status()
    got = kda_lib.recurrent_kda_backward(*(inp[n] for n in names), dout, None, dht,
                                         want_dh0=False, dev_status=st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    x = {n: inp[n].float() for n in names}
    gd = torch.Generator(device="cuda").manual_seed(12)
    d = {n: torch.randn(x[n].shape, generator=gd, device="cuda") for n in names}
    key = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta")
    want = sum(float((got[key[n]].double() * d[n].double()).sum()) for n in names)

    def loss(eps):
        o, ht = kda_lib.recurrent_kda(*(x[n] + eps * d[n] for n in names), None,
                                      output_final_state=True)
        return float((o.double() * dout.double()).sum() + (ht.double() * dht.double()).sum())

    eps = 2e-3
    fd = (loss(eps) - loss(-eps)) / (2 * eps)
    assert abs(fd - want) <= 1e-2 * abs(want), (fd, want)
