"""kda_recurrent_fwd against the fp64 oracle, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import kda_synth
from tests import parity

pytestmark = pytest.mark.gpu


def _small(seed, B=2, T=50, H=2, HV=4, K=64, V=64, dtype=torch.bfloat16, h0=True, g_hi=0.5):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, H, K, generator=gen)
    k = torch.randn(B, T, H, K, generator=gen)
    q, k = q / q.norm(dim=-1, keepdim=True), k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, HV, V, generator=gen)
    beta = torch.sigmoid(torch.randn(B, T, HV, generator=gen))
    g = -torch.rand(B, T, HV, K, generator=gen) * g_hi
    s = 0.1 * torch.randn(B, HV, K, V, generator=gen) if h0 else None
    d = dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), beta=beta.to(dtype), g=g, h0=s,
             cu_seqlens=None, N=B)
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in d.items()}


def _run(kda, inp, **kw):
    return kda.recurrent_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"],
                             cu_seqlens=inp["cu_seqlens"], output_final_state=True, **kw)


def _check(inp, o, ht, tol, **kw):
    ref = parity.oracle_forward(inp, **kw)
    e_o, e_h = parity.compare_sampled(inp, o, ht, ref, tol)
    assert e_o <= tol and e_h <= tol, (e_o, e_h)
    return e_o, e_h


def test_tiny_fp32_workload(kda_lib):
    inp = kda_synth.make_inputs(0, device="cuda")
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, parity.TOL[torch.float32])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (96, 100), (32, 256), (100, 7), (256, 130)])
def test_shapes(kda_lib, dtype, K, V):
    inp = _small(K * 1000 + V, K=K, V=V, dtype=dtype)
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, parity.TOL[dtype] if dtype == torch.bfloat16 else 1e-4)


def test_gva_and_l2norm_flag(kda_lib):
    inp = _small(7, H=2, HV=8, K=64, V=32, dtype=torch.float32)
    inp["q"] = inp["q"] * 3.0  # unnormalised rows: the flag must normalise them
    inp["k"] = inp["k"] * 0.5
    o, ht = _run(kda_lib, inp, use_qk_l2norm_in_kernel=True)
    _check(inp, o, ht, 1e-4, l2norm=True)


def test_scale_and_g_scale(kda_lib):
    inp = _small(8, dtype=torch.float32)
    o, ht = _run(kda_lib, inp, scale=0.3, g_scale=1.4426950408889634)
    _check(inp, o, ht, 1e-4, scale=0.3, g_scale=1.4426950408889634)


def test_no_h0_and_no_ht(kda_lib):
    inp = _small(9, h0=False)
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 2e-2)
    o2, ht2 = kda_lib.recurrent_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    assert ht2 is None and torch.equal(o, o2)


def test_ht_may_alias_h0(kda_lib):
    inp = _small(10, dtype=torch.float32)
    o_ref, ht_ref = _run(kda_lib, inp)
    state = inp["h0"].clone()
    o, ht = kda_lib.recurrent_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], state,
                                  final_state_out=state)
    assert torch.equal(o, o_ref) and torch.equal(state, ht_ref)


def _packed(seed, lens, HV=4, H=2, K=64, V=48, cap_extra=37, dtype=torch.bfloat16):
    total = sum(lens)
    T = total + cap_extra
    inp = _small(seed, B=1, T=T, H=H, HV=HV, K=K, V=V, dtype=dtype, h0=False)
    N = len(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    for name in ("q", "k", "v", "beta", "g"):
        inp[name][:, total:] = float("nan")
    gen = torch.Generator().manual_seed(seed + 1)
    inp["h0"] = (0.1 * torch.randn(N, HV, K, V, generator=gen)).cuda()
    inp["cu_seqlens"] = cu.cuda()
    inp["N"] = N
    return inp


def test_packed_empty_slots_and_nan_tail(kda_lib):
    lens = [5, 0, 64, 0, 0, 1, 130, 0]
    inp = _packed(11, lens)
    sentinel = 12345.0
    o = torch.full_like(inp["v"], sentinel)
    ht = torch.full_like(inp["h0"], sentinel)
    shape = kda_lib.make_shape(inp["q"], inp["v"], inp["cu_seqlens"])
    st = kda_lib.new_status()
    kda_lib.kda_recurrent_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"],
                              inp["cu_seqlens"], shape, o, ht, st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    _check(inp, o, ht, 2e-2)
    end = sum(lens)
    assert torch.all(o[:, end:] == sentinel), "rows beyond the terminal offset were written"
    for n, L in enumerate(lens):
        if L == 0:  # empty slot: bitwise passthrough
            assert torch.equal(ht[n].view(torch.int32), inp["h0"][n].view(torch.int32))


def test_packed_empty_slot_without_h0_is_positive_zero(kda_lib):
    inp = _packed(12, [3, 0, 4])
    inp["h0"] = None
    o, ht = _run(kda_lib, inp)
    assert torch.all(ht[1].view(torch.int32) == 0)


@pytest.mark.parametrize("bad", [[1, 3, 8], [0, 5, 3], [0, 3, 10 ** 6], [-4, 3, 8]])
def test_invalid_offsets_set_status_and_write_nothing(kda_lib, bad):
    inp = _packed(13, [3, 5])
    inp["cu_seqlens"] = torch.tensor(bad, dtype=torch.int32, device="cuda")
    sentinel = -777.0
    o = torch.full_like(inp["v"], sentinel)
    ht = torch.full_like(inp["h0"], sentinel)
    shape = kda_lib.make_shape(inp["q"], inp["v"], inp["cu_seqlens"])
    st = kda_lib.new_status()
    kda_lib.kda_recurrent_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"],
                              inp["cu_seqlens"], shape, o, ht, st)
    status, bits = kda_lib.kda_read_device_status(st)
    assert status == kda_lib.KDA_ERR_BAD_CU_SEQLENS and bits & 1
    # The slot whose own offsets are bad is skipped entirely.
    bad_slots = [n for n in range(2) if not (0 <= bad[n] <= bad[n + 1] <= inp["q"].shape[1]
                                             and (n > 0 or bad[0] == 0))]
    for n in bad_slots:
        assert torch.all(ht[n] == sentinel)


def test_decode_workload_dense_and_packed(kda_lib):
    """4096 sequences x 1 token x 32 heads: 131072 (sequence, head) programs on
    grid x; sampled sequences checked against the oracle; dense == packed."""
    inp = kda_synth.make_inputs(4, device="cuda")
    o, ht = _run(kda_lib, inp)
    seqs = [0, 1, 777, 2048, 4095]
    ref = parity.oracle_forward(inp, seqs=seqs)
    e_o, e_h = parity.compare_sampled(inp, o, ht, ref, 2e-2)
    assert e_o <= 2e-2 and e_h <= 2e-2, (e_o, e_h)
    pk = kda_synth.make_inputs(4, device="cuda", packed_decode=True)
    for name in ("q", "k", "v", "g", "beta", "h0"):
        assert torch.equal(pk[name].reshape(-1), inp[name].reshape(-1))
    o2, ht2 = _run(kda_lib, pk)
    assert torch.equal(o2.reshape(-1), o.reshape(-1)) and torch.equal(ht2, ht)


def test_decode_prefill_variant_256_tokens(kda_lib):
    """The 256-token prefill variant of the decode workload, full size, sampled."""
    w = kda_synth.workload(4, T=256)
    inp = kda_synth.make_inputs(w, device="cuda")
    o, ht = _run(kda_lib, inp)
    ref = parity.oracle_forward(inp, seqs=[0, 2999, 4095], heads=[0, 31])
    e_o, e_h = parity.compare_sampled(inp, o, ht, ref, 2e-2)
    assert e_o <= 2e-2 and e_h <= 2e-2, (e_o, e_h)


def test_bitwise_deterministic(kda_lib):
    inp = _small(14, T=40)
    a = _run(kda_lib, inp)
    b = _run(kda_lib, inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_extreme_decay_finite(kda_lib):
    inp = _small(15, dtype=torch.float32)
    inp["g"].fill_(-16.0)
    o, ht = _run(kda_lib, inp)
    assert torch.isfinite(o).all() and torch.isfinite(ht).all()
    _check(inp, o, ht, 1e-4)


def test_cuda_graph_replay_with_mutated_offsets(kda_lib):
    """Capture once, then mutate cu_seqlens and the inputs in place and replay."""
    inp = _packed(16, [10, 20, 0, 30], dtype=torch.float32)
    cu = inp["cu_seqlens"]
    shape = kda_lib.make_shape(inp["q"], inp["v"], cu)
    o = torch.zeros_like(inp["v"])
    ht = torch.zeros_like(inp["h0"])
    st = kda_lib.new_status()
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        kda_lib.kda_recurrent_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["h0"], cu, shape, o, ht, st, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kda_lib.kda_recurrent_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["h0"], cu, shape, o, ht, st, stream=s)
    for lens in ([10, 20, 0, 30], [0, 45, 5, 10], [1, 1, 1, 1]):
        cu.copy_(torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32))
        inp["v"].mul_(-1.0)
        o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        _check(inp, o, ht, 1e-4)


def _with_kernels(kda, fn):
    kda.kda_profile_reset()
    kda.kda_profile_enable(True)
    try:
        out = fn()
        torch.cuda.synchronize()
        rep = kda.kda_profile_report()
    finally:
        kda.kda_profile_enable(False)
    return out, rep


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [8, 16, 17, 33, 83])
def test_long_form_across_token_groups(kda_lib, dtype, T):
    """Slots of many tokens take the grouped form (16 tokens per staged group);
    lengths at and around the group size, and a ragged last group."""
    inp = _small(300 + T, B=2, T=T, H=2, HV=4, K=128, V=128, dtype=dtype)
    (o, ht), rep = _with_kernels(kda_lib, lambda: _run(kda_lib, inp))
    assert "recurrent_long" in rep, rep
    _check(inp, o, ht, parity.TOL[dtype])


def test_long_form_packed_group_boundaries_and_nan_tail(kda_lib):
    lens = [16, 17, 0, 1, 33, 47, 2, 0]
    inp = _packed(31, lens, HV=4, H=1, K=128, V=256)
    sentinel = 777.0
    o = torch.full_like(inp["v"], sentinel)
    ht = torch.full_like(inp["h0"], sentinel)
    shape = kda_lib.make_shape(inp["q"], inp["v"], inp["cu_seqlens"])
    st = kda_lib.new_status()
    _, rep = _with_kernels(kda_lib, lambda: kda_lib.kda_recurrent_fwd(
        inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"], inp["cu_seqlens"],
        shape, o, ht, st))
    assert "recurrent_long" in rep, rep
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    _check(inp, o, ht, 2e-2)
    end = sum(lens)
    assert torch.all(o[:, end:] == sentinel)
    for n, L in enumerate(lens):
        if L == 0:
            assert torch.equal(ht[n].view(torch.int32), inp["h0"][n].view(torch.int32))


def test_long_form_l2norm_and_small_k(kda_lib):
    inp = _small(41, B=1, T=70, H=1, HV=2, K=32, V=64, dtype=torch.float32)
    inp["q"] = inp["q"] * 2.0  # unnormalised rows: the flag must normalise them
    inp["k"] = inp["k"] * 0.7
    (o, ht), rep = _with_kernels(kda_lib, lambda: _run(kda_lib, inp, use_qk_l2norm_in_kernel=True))
    assert "recurrent_long" in rep, rep
    _check(inp, o, ht, 1e-4, l2norm=True)


def test_single_token_slots_take_the_register_exchange_form(kda_lib):
    inp = _small(42, B=8, T=1)
    (o, ht), rep = _with_kernels(kda_lib, lambda: _run(kda_lib, inp))
    assert "recurrent" in rep and "recurrent_long" not in rep, rep
    _check(inp, o, ht, 2e-2)


def test_long_and_short_forms_agree(kda_lib):
    """State columns are independent, so the first 60 value columns of a 64-column
    problem (grouped form) equal a 60-column problem, which bf16 rows of 120
    bytes send to the register-exchange form."""
    inp = _small(43, B=2, T=40, H=2, HV=2, K=64, V=64)
    (o1, ht1), rep1 = _with_kernels(kda_lib, lambda: _run(kda_lib, inp))
    assert "recurrent_long" in rep1
    cut = dict(inp)
    cut["v"] = inp["v"][..., :60].contiguous()
    cut["h0"] = inp["h0"][..., :60].contiguous()
    (o2, ht2), rep2 = _with_kernels(kda_lib, lambda: _run(kda_lib, cut))
    assert "recurrent" in rep2 and "recurrent_long" not in rep2, rep2
    assert parity.rel_err(ht1[..., :60], ht2) <= 1e-5
    assert parity.rel_err(o1[..., :60], o2) <= 8e-3
