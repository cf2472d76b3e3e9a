"""Split launches of the chunked forward (GPU, KDA_FLAG_SPLIT_SCAN): few long
sequences run each sequence's scan as two segments at once and compose them
afterwards (o_c += Q_c E0 over the second segment, ht = P E0 + E1).  Every case
here is a shape that takes the split; each is checked against the fp64 oracle
through the C ABI, and the launch is checked to have run the composition
kernel."""
import pytest
import torch

from tests import parity
from tests.test_gpu_recurrent import _packed, _small

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _run_profiled(kda, inp, split=True):
    kda.kda_profile_reset()
    kda.kda_profile_enable(True)
    try:
        o, ht = kda.chunk_kda(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              initial_state=inp["h0"], output_final_state=True,
                              cu_seqlens=inp["cu_seqlens"], split_scan=split)
        torch.cuda.synchronize()
        report = kda.kda_profile_report()
    finally:
        kda.kda_profile_enable(False)
    return o, ht, report


def _check_all(inp, o, ht):
    ref = parity.oracle_forward(inp)
    e_o, e_h = parity.compare_sampled(inp, o, ht, ref, TOL)
    assert e_o <= TOL and e_h <= TOL, (e_o, e_h)


@pytest.mark.parametrize("T,H,HV,K,V,h0", [
    (2085, 2, 2, 128, 128, True),   # ragged last chunk, initial state
    (1500, 1, 2, 64, 64, False),    # K = V = 64, two value heads per q/k head
    (1100, 1, 1, 128, 256, True),   # V = 256 (four 64-column blocks)
    (1024, 2, 2, 128, 192, True),   # even chunk count, V = 192
])
def test_split_dense(kda_lib, T, H, HV, K, V, h0):
    inp = _small(T + V, B=1, T=T, H=H, HV=HV, K=K, V=V, h0=h0)
    o, ht, rep = _run_profiled(kda_lib, inp)
    assert "chunk_fix_tc" in rep, rep
    _check_all(inp, o, ht)


def test_split_packed_with_empty_and_single_chunk_sequences(kda_lib):
    # sequences of 0 and 1 chunk leave the second segment empty (ht = E0 exactly)
    lens = [1500, 0, 64, 700, 1, 0, 1100]
    inp = _packed(77, lens, HV=2, H=1, K=128, V=128)
    cu = inp["cu_seqlens"]
    sentinel = 4321.0
    o = torch.full_like(inp["v"], sentinel)
    ht = torch.full_like(inp["h0"], sentinel)
    shape = kda_lib.make_shape(inp["q"], inp["v"], cu, flags=kda_lib.KDA_FLAG_SPLIT_SCAN)
    ws = torch.empty(kda_lib.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    st = kda_lib.new_status()
    kda_lib.kda_profile_reset()
    kda_lib.kda_profile_enable(True)
    try:
        kda_lib.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"], cu,
                              shape, o, ht, ws, st)
        torch.cuda.synchronize()
        rep = kda_lib.kda_profile_report()
    finally:
        kda_lib.kda_profile_enable(False)
    assert "chunk_fix_tc" in rep, rep
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    _check_all(inp, o, ht)
    end = int(cu[-1])
    assert torch.all(o[:, end:] == sentinel)
    for n, length in enumerate(lens):
        if length == 0:
            assert torch.equal(ht[n].view(torch.int32), inp["h0"][n].view(torch.int32))


def test_split_matches_unsplit_run(kda_lib):
    """The same call with and without KDA_FLAG_SPLIT_SCAN agrees within the bf16
    tolerance."""
    T, HV = 1536, 2
    inp = _small(5, B=1, T=T, H=2, HV=HV, K=128, V=128)
    o1, ht1, rep1 = _run_profiled(kda_lib, inp)
    assert "chunk_fix_tc" in rep1
    o2, ht2, rep2 = _run_profiled(kda_lib, inp, split=False)
    assert "chunk_fix_tc" not in rep2
    assert parity.rel_err(o1[0], o2[0]) <= TOL
    assert parity.rel_err(ht1[0], ht2[0]) <= TOL
