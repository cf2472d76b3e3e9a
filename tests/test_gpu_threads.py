"""Two host threads making their first kda_chunk_fwd calls at the same time.

The library sets kernel attributes and reads device limits once per device, on
the first call that needs them; two threads that arrive there together must
both get a correct launch.  The test runs in a fresh process (no earlier call
has done that setup): two threads, each with its own stream, inputs, workspace
and outputs, start at one barrier and call kda_chunk_fwd (one dense input that
takes the pipelined launch, one packed input).  Both results must match the
fp64 oracle within the bf16 tolerance, and equal bit for bit what the same
calls give when made one after the other afterwards.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import gated_delta_rule_cumsum_gb300 as kda
import kda_synth
from tests import parity

dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
kda.load()
cases = [
    kda_synth.make_inputs(kda_synth.workload(1, T=2048, H=4, HV=4, seed=31), device=dev),
    kda_synth.make_inputs(kda_synth.workload(3, n_seqs=6, n_empty=2, len_max=700,
                                             fill_limit=2000, T=2048, H=4, HV=4, seed=32),
                          device=dev),
]
torch.cuda.synchronize()
barrier = threading.Barrier(len(cases))
results, errors = [None] * len(cases), []

def run(i, inp, stream, wait):
    try:
        q, k, v, g, beta, h0, cu = (inp[n] for n in ("q", "k", "v", "g", "beta", "h0",
                                                     "cu_seqlens"))
        if wait:
            barrier.wait()
        shape = kda.make_shape(q, v, cu)
        ws = torch.empty(kda.kda_chunk_workspace_size(shape), dtype=torch.uint8, device=dev)
        o = torch.full_like(v, float("nan"))
        ht = torch.full((inp["N"], v.shape[2], q.shape[3], v.shape[3]), float("nan"),
                        device=dev)
        st = kda.new_status(dev)
        with torch.cuda.stream(stream):
            kda.kda_chunk_fwd(q, k, v, g, beta, h0, cu, shape, o, ht, ws, st, stream)
            assert kda.kda_read_device_status(st, stream) == (0, 0)
        results[i] = (o, ht)
    except BaseException as e:  # noqa: BLE001
        errors.append(repr(e))

streams = [torch.cuda.Stream(dev) for _ in cases]
threads = [threading.Thread(target=run, args=(i, c, s, True))
           for i, (c, s) in enumerate(zip(cases, streams))]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
concurrent = list(results)
for i, c in enumerate(cases):  # the same calls, one after the other
    run(i, c, streams[i], False)
assert not errors, errors
for i, inp in enumerate(cases):
    o, ht = concurrent[i]
    same = lambda a, b: torch.allclose(a, b, rtol=0, atol=0, equal_nan=True)  # NaN: untouched rows
    assert same(o, results[i][0]) and same(ht, results[i][1]), f"case {i}"
    tol = parity.TOL[torch.bfloat16]
    e_o, e_h = parity.compare_sampled(inp, o, ht, parity.oracle_forward(inp), tol)
    assert e_o <= tol and e_h <= tol, (i, e_o, e_h)
print("threads ok")
"""


def test_two_threads_first_calls_at_once_in_a_fresh_process(kda_lib):
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
