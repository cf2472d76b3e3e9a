"""kda_gate_cumsum against the fp64 oracle, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import kda_synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chunk", [1, 16, 63, 64])
def test_dense(kda_lib, chunk):
    g = -torch.rand(3, 200, 5, 64, generator=torch.Generator().manual_seed(chunk))
    got = kda_lib.gate_cumsum(g.cuda(), chunk_size=chunk, g_scale=1.3)
    want = oracle.gate_cumsum(g, chunk=chunk, g_scale=1.3)
    assert parity.rel_err(got, want) <= 1e-5


def test_packed_workload(kda_lib):
    inp = kda_synth.make_inputs(3, device="cuda")
    cu = inp["cu_seqlens"]
    st = kda_lib.new_status()
    got = kda_lib.gate_cumsum(inp["g"], cu_seqlens=cu, chunk_size=64, dev_status=st)
    assert kda_lib.kda_read_device_status(st) == (0, 0)
    end = int(cu[-1])
    g_cpu = inp["g"][:, : end + 64].cpu()
    want = oracle.gate_cumsum(g_cpu, cu_seqlens=cu.cpu(), chunk=64)
    assert parity.rel_err(got[:, :end], want[:, :end]) <= 1e-5
    assert torch.all(got[:, end:] == 0), "tail rows must not be written"


def test_chunk_one_is_identity(kda_lib):
    g = -torch.rand(1, 77, 2, 128).cuda()
    assert torch.equal(kda_lib.gate_cumsum(g, chunk_size=1), g)


def test_invalid_offsets_reported(kda_lib):
    g = -torch.rand(1, 100, 2, 64).cuda()
    st = kda_lib.new_status()
    cu = torch.tensor([0, 50, 40, 100], dtype=torch.int32, device="cuda")
    kda_lib.gate_cumsum(g, cu_seqlens=cu, dev_status=st)
    status, bits = kda_lib.kda_read_device_status(st)
    assert status == kda_lib.KDA_ERR_BAD_CU_SEQLENS
