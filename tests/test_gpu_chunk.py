"""kda_chunk_fwd against the fp64 oracle, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import kda_synth
from tests import parity
from tests.test_gpu_recurrent import _packed, _small

pytestmark = pytest.mark.gpu


def _run(kda, inp, **kw):
    return kda.chunk_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                         initial_state=inp["h0"], output_final_state=True,
                         cu_seqlens=inp["cu_seqlens"], **kw)


def _check(inp, o, ht, tol, **kw):
    ref = parity.oracle_forward(inp, **{k: v for k, v in kw.items() if k in ("heads", "seqs",
                                                                               "l2norm", "scale",
                                                                               "g_scale")})
    e_o, e_h = parity.compare_sampled(inp, o, ht, ref, tol)
    assert e_o <= tol and e_h <= tol, (e_o, e_h)
    return e_o, e_h


def test_tiny_fp32_workload(kda_lib):
    inp = kda_synth.make_inputs(0, device="cuda")
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 1e-4)


def test_training_shape_workload(kda_lib):
    """B1 T8192 H=HV16 K=V128 bf16, h0 = 0, final state stored: every head, in the
    launch configuration the benchmark times (pipelined: two preps, two scans)."""
    inp = kda_synth.make_inputs(1, device="cuda")
    kda_lib.kda_profile_reset()
    kda_lib.kda_profile_enable(True)
    try:
        o, ht = _run(kda_lib, inp)
        torch.cuda.synchronize()
        rep = kda_lib.kda_profile_report()
    finally:
        kda_lib.kda_profile_enable(False)
    assert rep["chunk_prep_tc"][1] == 2 and rep["chunk_scan_tc"][1] == 2, rep
    _check(inp, o, ht, 2e-2)


def test_grouped_value_heads_workload(kda_lib):
    """B4 T4096 H8 HV32 (4 value heads per q/k head): sampled (batch, head) pairs."""
    inp = kda_synth.make_inputs(2, device="cuda")
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 2e-2, seqs=[0, 3], heads=[0, 5, 7])


def test_packed_varlen_workload(kda_lib):
    """64 geometric-length sequences + 8 empty slots, NaN tail below capacity."""
    inp = kda_synth.make_inputs(3, device="cuda")
    cu = inp["cu_seqlens"]
    sentinel = 4242.0
    o = torch.full_like(inp["v"], sentinel)
    ht = torch.full((inp["N"], 32, 128, 128), sentinel, device="cuda")
    shape = kda_lib.make_shape(inp["q"], inp["v"], cu)
    ws = torch.empty(kda_lib.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    st = kda_lib.new_status()
    kda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"], cu,
                          shape, o, ht, ws, st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    _check(inp, o, ht, 2e-2, heads=[0, 13, 31])
    end = int(cu[-1])
    assert torch.all(o[:, end:] == sentinel)
    cl = cu.cpu().tolist()
    empties = [n for n in range(inp["N"]) if cl[n] == cl[n + 1]]
    assert len(empties) == 8
    for n in empties:
        assert torch.equal(ht[n].view(torch.int32), inp["h0"][n].view(torch.int32))


@pytest.mark.parametrize("K,V,T,lens", [
    (32, 64, 300, None),             # padded to the 64-channel kernels
    (8, 32, 200, None),
    (96, 128, 700, None),            # padded to the 128-channel kernels
    (72, 96, 0, [450, 0, 70, 129]),  # packed, an empty slot
    (120, 256, 0, [333, 64]),
])
def test_tensor_core_path_any_k_multiple_of_8(kda_lib, K, V, T, lens):
    """bf16 K not in {64, 128}: the tensor-core kernels with zero channels past K."""
    if lens is None:
        inp = _small(K * 10 + V, B=2, T=T, H=2, HV=4, K=K, V=V)
    else:
        inp = _packed(K + V, lens, HV=2, H=1, K=K, V=V)
    kda_lib.kda_profile_reset()
    kda_lib.kda_profile_enable(True)
    try:
        o, ht = _run(kda_lib, inp)
        torch.cuda.synchronize()
        rep = kda_lib.kda_profile_report()
    finally:
        kda_lib.kda_profile_enable(False)
    assert "chunk_prep_tc" in rep, rep
    _check(inp, o, ht, 2e-2)
    if lens is not None:
        for n, L in enumerate(lens):
            if L == 0:
                assert torch.equal(ht[n].view(torch.int32), inp["h0"][n].view(torch.int32))


def test_wide_scan_two_ctas_per_head(kda_lib):
    """128 value columns per scan CTA with two CTAs per (sequence, head): B=2, HV=48,
    V=256 is 384 CTAs of 64 columns, more than one wave of SMs, and chunks with a
    ragged tail (T=200)."""
    inp = _small(77, B=2, T=200, H=16, HV=48, K=128, V=256)
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 2e-2, heads=[0, 7, 15])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K,V,T", [(64, 64, 1), (64, 16, 63), (128, 96, 64), (128, 256, 65),
                                   (64, 128, 200), (128, 40, 130), (128, 64, 100)])
def test_shapes(kda_lib, dtype, K, V, T):
    inp = _small(K + V + T, B=2, T=T, K=K, V=V, dtype=dtype)
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 1e-4 if dtype == torch.float32 else 2e-2)


def test_no_h0_no_ht_and_alias(kda_lib):
    inp = _small(3, T=100, dtype=torch.float32)
    o_ref, ht_ref = _run(kda_lib, inp)
    o2, ht2 = kda_lib.chunk_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                initial_state=inp["h0"])
    assert ht2 is None and torch.equal(o2, o_ref)
    # ht aliasing h0 (in-place state update)
    state = inp["h0"].clone()
    shape = kda_lib.make_shape(inp["q"], inp["v"])
    ws = torch.empty(kda_lib.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o3 = torch.empty_like(inp["v"])
    kda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], state, None, shape,
                          o3, state, ws)
    assert torch.equal(o3, o_ref) and torch.equal(state, ht_ref)
    inp["h0"] = None
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 1e-4)


def test_gate_cumsum_input_flag(kda_lib):
    """g given as the chunk-local cumsum (kda_gate_cumsum output) gives the same result."""
    inp = _packed(5, [70, 0, 129, 64], dtype=torch.float32)
    o_ref, ht_ref = _run(kda_lib, inp)
    gc = kda_lib.gate_cumsum(inp["g"], cu_seqlens=inp["cu_seqlens"], chunk_size=64)
    inp2 = dict(inp, g=gc)
    o, ht = _run(kda_lib, inp2, g_is_cumsum=True)
    end = int(inp["cu_seqlens"][-1])
    assert parity.rel_err(o[:, :end], o_ref[:, :end]) <= 1e-5
    assert parity.rel_err(ht, ht_ref) <= 1e-5


def test_l2norm_flag(kda_lib):
    inp = _small(6, T=90, dtype=torch.float32)
    inp["q"] = inp["q"] * 2.5
    inp["k"] = inp["k"] * 0.3
    o, ht = _run(kda_lib, inp, use_qk_l2norm_in_kernel=True)
    _check(inp, o, ht, 1e-4, l2norm=True)


def test_extreme_decay(kda_lib):
    """g = -16 per step (ALGORITHM.md's guard case): finite and on the oracle."""
    inp = _small(7, T=130, dtype=torch.float32)
    inp["g"].fill_(-16.0)
    o, ht = _run(kda_lib, inp)
    assert torch.isfinite(o).all() and torch.isfinite(ht).all()
    _check(inp, o, ht, 1e-4)


@pytest.mark.parametrize("lo,hi", [(0.8, 1.6), (1.5, 3.0)])
def test_wide_gate_range_chunks(kda_lib, lo, hi):
    """Per-token gates of -U(lo, hi) (log2): chunk gate ranges of about 77 and 144, past
    the split grams' limit, so every chunk's grams are formed exactly; several chunks,
    a ragged tail, two value heads per q/k head."""
    inp = _small(31, B=1, T=300, H=1, HV=2, K=128, V=128, dtype=torch.bfloat16)
    gen = torch.Generator().manual_seed(32)
    inp["g"] = -(lo + (hi - lo) * torch.rand(inp["g"].shape, generator=gen)).cuda()
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 2e-2)


def _wide_gates(inp, seed, rows=None):
    """-U(1.5, 3) log2 per token and channel (a chunk's range about 144) in the first
    `rows` rows (all by default); the rest keep what they hold."""
    g = inp["g"]
    rows = g.shape[1] if rows is None else rows
    gen = torch.Generator().manual_seed(seed)
    w = -(1.5 + 1.5 * torch.rand((g.shape[0], rows) + tuple(g.shape[2:]), generator=gen))
    g[:, :rows] = w.to(g.device)


@pytest.mark.parametrize("K,V", [(64, 64), (64, 128), (128, 256)])
def test_wide_gate_other_tile_sizes(kda_lib, K, V):
    """Every chunk on the exact grams with 64-channel tiles (their tensor-core operand
    then sits where L is later written) and with 256 value columns (inside v's region):
    several chunks, a ragged tail, two value heads per q/k head."""
    inp = _small(33, B=1, T=200, H=1, HV=2, K=K, V=V, dtype=torch.bfloat16)
    _wide_gates(inp, 34)
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 2e-2)


def test_wide_gate_packed(kda_lib):
    """The exact grams on packed sequences: short and empty slots, chunks that end
    inside a sequence's last rows, a NaN tail past the last offset."""
    lens = [1, 0, 63, 64, 65, 0, 130, 7]
    inp = _packed(35, lens, HV=2, H=1, K=128, V=128, dtype=torch.bfloat16)
    _wide_gates(inp, 36, rows=sum(lens))
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 2e-2)


def test_extreme_decay_bf16(kda_lib):
    """g = -16 per step on the bf16 tensor-core path: every boundary factor past a few
    rows underflows to zero, and the result is still the oracle's."""
    inp = _small(37, B=1, T=130, H=1, HV=2, K=128, V=128, dtype=torch.bfloat16)
    inp["g"].fill_(-16.0)
    o, ht = _run(kda_lib, inp)
    assert torch.isfinite(o).all() and torch.isfinite(ht).all()
    _check(inp, o, ht, 2e-2)


def test_mixed_extreme_and_mild_channels(kda_lib):
    inp = _small(8, T=128, K=128, V=64, dtype=torch.bfloat16)
    inp["g"][..., ::3] = -20.0
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 2e-2)


def test_packed_edge_cases(kda_lib):
    lens = [1, 0, 63, 64, 65, 0, 128, 200, 0]
    inp = _packed(9, lens, HV=4, H=1, K=64, V=64, dtype=torch.float32)
    o, ht = _run(kda_lib, inp)
    _check(inp, o, ht, 1e-4)


@pytest.mark.parametrize("bad", [[1, 3, 8], [0, 5, 3], [0, 3, 10 ** 6]])
def test_invalid_offsets(kda_lib, bad):
    inp = _packed(10, [3, 5])
    inp["cu_seqlens"] = torch.tensor(bad, dtype=torch.int32, device="cuda")
    sentinel = -5.0
    o = torch.full_like(inp["v"], sentinel)
    ht = torch.full_like(inp["h0"], sentinel)
    shape = kda_lib.make_shape(inp["q"], inp["v"], inp["cu_seqlens"])
    ws = torch.empty(kda_lib.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    st = kda_lib.new_status()
    kda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"],
                          inp["cu_seqlens"], shape, o, ht, ws, st)
    status, bits = kda_lib.kda_read_device_status(st)
    assert status == kda_lib.KDA_ERR_BAD_CU_SEQLENS
    assert torch.all(o == sentinel) and torch.all(ht == sentinel)


def test_guard_bands_untouched(kda_lib):
    """Outputs sit inside larger buffers; the canaries around them survive."""
    inp = _packed(11, [17, 0, 90])
    T, HV, V = inp["v"].shape[1], inp["v"].shape[2], inp["v"].shape[3]
    pad = 4096
    obuf = torch.full((pad + T * HV * V + pad,), 9.0, dtype=torch.bfloat16, device="cuda")
    o = obuf[pad:pad + T * HV * V].view(1, T, HV, V)
    N, K = inp["N"], inp["q"].shape[3]
    hbuf = torch.full((pad + N * HV * K * V + pad,), 7.0, device="cuda")
    ht = hbuf[pad:pad + N * HV * K * V].view(N, HV, K, V)
    shape = kda_lib.make_shape(inp["q"], inp["v"], inp["cu_seqlens"])
    ws = torch.empty(kda_lib.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    kda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"],
                          inp["cu_seqlens"], shape, o, ht, ws)
    torch.cuda.synchronize()
    assert torch.all(obuf[:pad] == 9.0) and torch.all(obuf[-pad:] == 9.0)
    assert torch.all(hbuf[:pad] == 7.0) and torch.all(hbuf[-pad:] == 7.0)
    _check(inp, o, ht, 2e-2)


def test_chunked_equals_recurrent_kernel(kda_lib):
    """The two kernels agree with each other on the same inputs (fp32)."""
    inp = _packed(12, [100, 0, 257], dtype=torch.float32)
    o1, h1 = _run(kda_lib, inp)
    o2, h2 = kda_lib.recurrent_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                   inp["h0"], cu_seqlens=inp["cu_seqlens"],
                                   output_final_state=True)
    end = int(inp["cu_seqlens"][-1])
    assert parity.rel_err(o1[:, :end], o2[:, :end]) <= 1e-5
    assert parity.rel_err(h1, h2) <= 1e-5


def test_prefill_then_decode_continuation(kda_lib):
    """chunk on tokens [0, 150) then recurrent on [150, 160) == oracle on [0, 160)."""
    inp = _small(13, B=1, T=160, dtype=torch.float32)
    pre = {n: (t[:, :150] if n in ("q", "k", "v", "g", "beta") else t) for n, t in inp.items()}
    o1, h1 = _run(kda_lib, pre)
    o2, h2 = kda_lib.recurrent_kda(inp["q"][:, 150:], inp["k"][:, 150:], inp["v"][:, 150:],
                                   inp["g"][:, 150:], inp["beta"][:, 150:], h1,
                                   output_final_state=True)
    ref = parity.oracle_forward(inp)
    o_ref, h_ref = ref[(0, 0)]
    assert parity.rel_err(torch.cat([o1, o2], 1)[0, :, 0], o_ref) <= 1e-4
    assert parity.rel_err(h2[0, 0], h_ref) <= 1e-4


def test_bitwise_deterministic(kda_lib):
    inp = _small(14, T=300)
    a = _run(kda_lib, inp)
    b = _run(kda_lib, inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_cuda_graph_replay_with_mutated_offsets(kda_lib):
    inp = _packed(15, [64, 100, 0, 36], dtype=torch.float32)
    cu = inp["cu_seqlens"]
    shape = kda_lib.make_shape(inp["q"], inp["v"], cu)
    ws = torch.empty(kda_lib.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o = torch.zeros_like(inp["v"])
    ht = torch.zeros_like(inp["h0"])
    s = torch.cuda.Stream()
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"], cu, shape, o, ht, ws)
    with torch.cuda.stream(s):
        kda_lib.kda_chunk_fwd(*args, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kda_lib.kda_chunk_fwd(*args, stream=s)
    for lens in ([64, 100, 0, 36], [0, 1, 199, 0], [50, 50, 50, 50]):
        cu.copy_(torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32))
        inp["k"].mul_(-1.0)
        graph.replay()
        torch.cuda.synchronize()
        _check(inp, o, ht, 1e-4)
