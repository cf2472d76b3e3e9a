"""kda_chunk_fwd_noalloc, the entry point for callers that cannot allocate
device memory at call time, against kda_chunk_fwd with a caller workspace: the
same kernels run in the same order, so the outputs must agree bit for bit, on
two calls in a row that share the built-in scratch array.

Collected last on purpose (the zz prefix): if it fails, a run that stops at the
first failure has already run every other test.  It passes both alone in a
fresh process and after the other tests, since the entry point sets itself up
on its first call on a device.
"""
import pytest
import torch

from tests import parity
from tests.test_gpu_recurrent import _packed, _small

pytestmark = pytest.mark.gpu


def _reference(kda, inp, cu):
    # serial launches, as the no-alloc entry point runs them: the same kernels in
    # the same order, so the results must agree bit for bit
    shape = kda.make_shape(inp["q"], inp["v"], cu, flags=kda.KDA_FLAG_SERIAL)
    ws = torch.empty(kda.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(inp["v"])
    ht = torch.empty(shape.num_seqs, shape.HV, shape.K, shape.V, device="cuda")
    kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["h0"], cu, shape,
                      o, ht, ws)
    return o, ht, shape


@pytest.mark.parametrize("packed", [False, True])
def test_noalloc_matches_workspace_entry_point_twice(kda_lib, packed):
    if packed:
        inp = _packed(21, [100, 0, 257, 64], HV=4, H=2, K=128, V=128)
    else:
        inp = _small(22, B=2, T=300, H=2, HV=4, K=128, V=128)
    cu = inp["cu_seqlens"]
    o_ref, ht_ref, shape = _reference(kda_lib, inp, cu)
    assert kda_lib.kda_chunk_workspace_size(shape) <= kda_lib.KDA_NOALLOC_SCRATCH_BYTES
    end = int(cu[-1]) if cu is not None else inp["q"].shape[1]
    for _ in range(2):  # two calls in a row share the scratch array
        o = torch.full_like(inp["v"], float("nan"))
        ht = torch.full_like(ht_ref, float("nan"))
        st = kda_lib.new_status()
        kda_lib.kda_chunk_fwd_noalloc(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                      inp["h0"], cu, shape, o, ht, st)
        assert kda_lib.kda_read_device_status(st) == (0, 0)
        # bit for bit: a tolerance would hide scratch left over from the previous call
        assert torch.equal(o[:, :end], o_ref[:, :end])
        assert torch.equal(ht, ht_ref)
        assert parity.rel_err(o[:, :end], o_ref[:, :end]) == 0.0


def test_noalloc_rejects_shapes_beyond_its_scratch(kda_lib):
    big = kda_lib.KdaShape(1, 1 << 16, 16, 16, 128, 128, 1, 1, -1.0, 1.0, 0)
    assert kda_lib.kda_chunk_workspace_size(big) > kda_lib.KDA_NOALLOC_SCRATCH_BYTES
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kda_lib.KdaError) as err:
        kda_lib.kda_chunk_fwd_noalloc(x, x, x, x, x, None, None, big, x, None)
    assert err.value.status == kda_lib.KDA_ERR_UNSUPPORTED
    assert "scratch" in str(err.value)
