"""Pipelined launches of the chunked forward (GPU).  A dense bf16 call whose scan
leaves most SMs idle runs in two parts: the prep of every sequence's first
chunks, then that part's scan (final state to the workspace) while the prep of
the remaining chunks fills the other SMs from the library's side stream, then
the second part's scan from that state.  Each case here is a shape the plan
pipelines; the profile report must show two prep and two scan launches, so a
change of the plan cannot turn these into serial runs unseen."""
import pytest
import torch

from tests import parity
from tests.test_gpu_recurrent import _small

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _run(kda, inp, serial=False, **kw):
    kda.kda_profile_reset()
    kda.kda_profile_enable(True)
    try:
        o, ht = kda.chunk_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              initial_state=inp["h0"], output_final_state=True,
                              cu_seqlens=inp["cu_seqlens"], serial=serial, **kw)
        torch.cuda.synchronize()
        rep = kda.kda_profile_report()
    finally:
        kda.kda_profile_enable(False)
    return o, ht, rep


def _launches(rep, name):
    return rep[name][1] if name in rep else 0


def _assert_pipelined(rep):
    assert _launches(rep, "chunk_prep_tc") == 2 and _launches(rep, "chunk_scan_tc") == 2, rep


@pytest.mark.parametrize("B,T,HV,K,V,h0", [
    (1, 8229, 4, 128, 128, True),   # ragged last chunk, initial state
    (2, 4096, 4, 128, 128, False),  # two sequences
    (1, 8229, 4, 64, 64, True),     # K = V = 64
    (1, 8229, 4, 96, 128, True),    # K = 96 (zero channels past K)
])
def test_pipelined_matches_oracle(kda_lib, B, T, HV, K, V, h0):
    inp = _small(900 + T + K, B=B, T=T, H=HV, HV=HV, K=K, V=V, h0=h0)
    o, ht, rep = _run(kda_lib, inp)
    _assert_pipelined(rep)
    ref = parity.oracle_forward(inp)
    e_o, e_h = parity.compare_sampled(inp, o, ht, ref, TOL)
    assert e_o <= TOL and e_h <= TOL, (e_o, e_h)


def test_pipelined_agrees_with_serial(kda_lib):
    inp = _small(41, B=1, T=8229, H=2, HV=4, K=128, V=128)
    o1, ht1, rep1 = _run(kda_lib, inp)
    _assert_pipelined(rep1)
    o2, ht2, rep2 = _run(kda_lib, inp, serial=True)
    assert _launches(rep2, "chunk_prep_tc") == 1 and _launches(rep2, "chunk_scan_tc") == 1, rep2
    assert parity.rel_err(o1, o2) <= TOL and parity.rel_err(ht1, ht2) <= TOL


def test_pipelined_final_state_may_alias_initial_state(kda_lib):
    inp = _small(42, B=1, T=8229, H=4, HV=4, K=128, V=128)
    ref = parity.oracle_forward(inp)
    state = inp["h0"].clone()
    shape = kda_lib.make_shape(inp["q"], inp["v"], None)
    ws = torch.empty(kda_lib.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(inp["v"])
    st = kda_lib.new_status()
    kda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], state, None, shape,
                          o, state, ws, st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    e_o, e_h = parity.compare_sampled(inp, o, state, ref, TOL)
    assert e_o <= TOL and e_h <= TOL, (e_o, e_h)


def test_pipelined_with_fused_activations(kda_lib):
    from tests.test_gpu_activation import RCP_LN2, _check, _oracle_inputs, _raw

    inp = _small(43, B=1, T=8229, H=4, HV=4, K=128, V=128)
    g_raw, b_raw, A_log, dt_bias = _raw(inp, 43)
    o, ht, rep = _run(kda_lib, dict(inp, g=g_raw, beta=b_raw), g_scale=RCP_LN2, A_log=A_log,
                      dt_bias=dt_bias, beta_sigmoid_scale=2.0)
    _assert_pipelined(rep)
    _check(inp, _oracle_inputs(inp, g_raw, b_raw, A_log, dt_bias, 2.0), o, ht, TOL)


def test_pipelined_call_replays_in_a_cuda_graph(kda_lib):
    """The fork to the library's side stream and the join back are captured with
    the caller's stream; replays reproduce the eager result bit for bit."""
    inp = _small(44, B=1, T=8229, H=4, HV=4, K=128, V=128)
    shape = kda_lib.make_shape(inp["q"], inp["v"], None)
    ws = torch.empty(kda_lib.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(inp["v"])
    ht = torch.empty_like(inp["h0"])
    st = kda_lib.new_status()
    s = torch.cuda.Stream()
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"], None, shape, o, ht,
            ws, st)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        kda_lib.kda_chunk_fwd(*args, stream=s)  # eager first: creates the side stream
    torch.cuda.synchronize()
    o_eager, ht_eager = o.clone(), ht.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kda_lib.kda_chunk_fwd(*args, stream=s)
    for _ in range(2):
        o.fill_(float("nan"))
        ht.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_eager) and torch.equal(ht, ht_eager)
    assert kda_lib.kda_read_device_status(st) == (0, 0)


def test_pipelined_without_final_state_and_with_l2norm(kda_lib):
    """No final state stored (the first part's state still travels in the workspace)
    and the q/k L2 norm applied inside, in both parts."""
    inp = _small(45, B=1, T=8229, H=4, HV=4, K=128, V=128)
    inp["q"] = (inp["q"].float() * 3.0).to(inp["q"].dtype)  # unnormalised rows
    inp["k"] = (inp["k"].float() * 0.5).to(inp["k"].dtype)
    kda_lib.kda_profile_reset()
    kda_lib.kda_profile_enable(True)
    try:
        o, ht = kda_lib.chunk_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  initial_state=inp["h0"], output_final_state=False,
                                  use_qk_l2norm_in_kernel=True)
        torch.cuda.synchronize()
        rep = kda_lib.kda_profile_report()
    finally:
        kda_lib.kda_profile_enable(False)
    assert ht is None
    _assert_pipelined(rep)
    ref = parity.oracle_forward(inp, l2norm=True)
    e_o, _ = parity.compare_sampled(inp, o, None, ref, TOL)
    assert e_o <= TOL, e_o
