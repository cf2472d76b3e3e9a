"""A bounded on-device wait that runs out reports KDA_DEVICE_TIMEOUT, and the
context stays usable.

The scan kernel's waits all carry a time limit; when one gives up, the kernel
sets KDA_DEVICE_TIMEOUT in the caller's status word, issues no further MMA,
drains its own copies in flight (bounded) and returns.  KDA_FLAG_TEST_WAIT_TIMEOUT
makes the MMA issuer wait on a barrier nothing signals, with a 2 us limit, so
that path runs on every such call.  No GPU fault is involved: the wait is a
bounded poll of a shared-memory barrier.
"""
import pytest
import torch

import kda_synth
from tests import parity

pytestmark = pytest.mark.gpu


def _call(kda, inp, flags):
    q, k, v, g, beta, h0, cu = (inp[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"))
    shape = kda.make_shape(q, v, cu, flags=flags)
    ws = torch.empty(kda.kda_chunk_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o = torch.zeros_like(v)
    ht = torch.zeros(inp["N"], v.shape[2], q.shape[3], v.shape[3], device="cuda")
    st = kda.new_status()
    kda.kda_chunk_fwd(q, k, v, g, beta, h0, cu, shape, o, ht, ws, st)
    return kda.kda_read_device_status(st), o, ht


@pytest.mark.parametrize("serial", [True, False])
def test_wait_that_runs_out_reports_timeout_then_next_call_is_correct(kda_lib, serial):
    inp = kda_synth.make_inputs(kda_synth.workload(1, T=1536, H=2, HV=4, seed=41), device="cuda")
    base = kda_lib.KDA_FLAG_SERIAL if serial else 0
    (st, bits), _, _ = _call(kda_lib, inp, base | kda_lib.KDA_FLAG_TEST_WAIT_TIMEOUT)
    assert st == kda_lib.KDA_ERR_TIMEOUT and bits == kda_lib.KDA_DEVICE_TIMEOUT, (st, bits)
    # the same context, a normal call: no error, results at parity
    (st, bits), o, ht = _call(kda_lib, inp, base)
    assert (st, bits) == (kda_lib.KDA_OK, 0)
    tol = parity.TOL[torch.bfloat16]
    e_o, e_h = parity.compare_sampled(inp, o, ht, parity.oracle_forward(inp), tol)
    assert e_o <= tol and e_h <= tol, (e_o, e_h)
