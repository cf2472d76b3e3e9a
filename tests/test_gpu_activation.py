"""The input activations applied inside the op (the *_act entry points): the raw
gate through -exp(A_log) softplus(g + dt_bias) (natural log, times g_scale =
1/ln 2) and beta through sigmoid times 1 or 2, against the fp64 oracle applied
to the oracle's own activation of the same raw inputs (GPU)."""
import math

import numpy as np
import pytest
import torch

from oracle import activation as oact
from tests import parity
from tests.test_gpu_recurrent import _packed, _small

pytestmark = pytest.mark.gpu

RCP_LN2 = 1.0 / math.log(2.0)


def _raw(inp, seed):
    """Raw gate and beta logits for the shapes of `inp`, plus A_log, dt_bias."""
    gen = torch.Generator().manual_seed(seed)
    B, T, HV, K = inp["g"].shape
    g_raw = (torch.randn(B, T, HV, K, generator=gen) - 2.0).cuda()
    b_raw = torch.randn(B, T, HV, generator=gen).to(inp["beta"].dtype).cuda()
    A_log = torch.log(1.0 + 3.0 * torch.rand(HV, generator=gen)).cuda()
    dt_bias = (0.5 * torch.randn(HV, K, generator=gen)).cuda()
    return g_raw, b_raw, A_log, dt_bias


def _oracle_inputs(inp, g_raw, b_raw, A_log, dt_bias, beta_scale):
    """The inputs with g and beta replaced by the oracle's activation of the raw ones."""
    ref = dict(inp)
    ref["g"] = torch.from_numpy(oact.gate(g_raw, A_log, dt_bias))
    bf16 = inp["beta"].dtype == torch.bfloat16
    ref["beta"] = torch.from_numpy(oact.beta(b_raw, beta_scale, bf16=bf16))
    return ref


def _check(inp, ref, o, ht, tol):
    want = parity.oracle_forward(ref, g_scale=RCP_LN2)
    e_o, e_h = parity.compare_sampled(inp, o, ht, want, tol)
    assert e_o <= tol and e_h <= tol, (e_o, e_h)


@pytest.mark.parametrize("dtype,K,V,T,beta_scale", [
    (torch.bfloat16, 128, 128, 200, 2.0),   # tensor-core path, ragged last chunk
    (torch.bfloat16, 64, 64, 130, 1.0),
    (torch.float32, 64, 48, 150, 2.0),      # fp32 chunk path
])
def test_chunk_with_activations(kda_lib, dtype, K, V, T, beta_scale):
    inp = _small(T + K, B=2, T=T, K=K, V=V, dtype=dtype)
    g_raw, b_raw, A_log, dt_bias = _raw(inp, T)
    o, ht = kda_lib.chunk_kda(inp["q"], inp["k"], inp["v"], g_raw, b_raw,
                              initial_state=inp["h0"], output_final_state=True, g_scale=RCP_LN2,
                              A_log=A_log, dt_bias=dt_bias, beta_sigmoid_scale=beta_scale)
    ref = _oracle_inputs(inp, g_raw, b_raw, A_log, dt_bias, beta_scale)
    _check(inp, ref, o, ht, 2e-2 if dtype == torch.bfloat16 else 1e-4)


def test_chunk_activations_packed_and_split(kda_lib):
    lens = [1100, 0, 70]
    inp = _packed(31, lens, HV=2, H=1, K=128, V=128)
    g_raw, b_raw, A_log, dt_bias = _raw(inp, 31)
    for split in (False, True):
        o, ht = kda_lib.chunk_kda(inp["q"], inp["k"], inp["v"], g_raw, b_raw,
                                  initial_state=inp["h0"], output_final_state=True,
                                  cu_seqlens=inp["cu_seqlens"], g_scale=RCP_LN2, A_log=A_log,
                                  dt_bias=dt_bias, beta_sigmoid_scale=2.0, split_scan=split)
        ref = _oracle_inputs(inp, g_raw, b_raw, A_log, dt_bias, 2.0)
        _check(inp, ref, o, ht, 2e-2)
        assert torch.equal(ht[1].view(torch.int32), inp["h0"][1].view(torch.int32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_recurrent_with_activations(kda_lib, dtype):
    inp = _small(9, B=2, T=90, K=64, V=80, dtype=dtype)
    g_raw, b_raw, A_log, dt_bias = _raw(inp, 9)
    o, ht = kda_lib.recurrent_kda(inp["q"], inp["k"], inp["v"], g_raw, b_raw, inp["h0"],
                                  output_final_state=True, g_scale=RCP_LN2, A_log=A_log,
                                  dt_bias=dt_bias, beta_sigmoid_scale=1.0)
    ref = _oracle_inputs(inp, g_raw, b_raw, A_log, dt_bias, 1.0)
    _check(inp, ref, o, ht, 2e-2 if dtype == torch.bfloat16 else 1e-4)


def test_activation_without_bias_and_gate_only(kda_lib):
    """dt_bias NULL (no bias), and the gate activation alone (beta as given)."""
    inp = _small(4, B=1, T=100, K=128, V=128)
    g_raw, _, A_log, _ = _raw(inp, 4)
    o, ht = kda_lib.chunk_kda(inp["q"], inp["k"], inp["v"], g_raw, inp["beta"],
                              initial_state=inp["h0"], output_final_state=True, g_scale=RCP_LN2,
                              A_log=A_log)
    ref = dict(inp)
    ref["g"] = torch.from_numpy(oact.gate(g_raw, A_log))
    _check(inp, ref, o, ht, 2e-2)


@pytest.mark.parametrize("chunk", [1, 64])
def test_gate_cumsum_with_activation(kda_lib, chunk):
    inp = _small(12, B=2, T=150, K=64, V=16, dtype=torch.float32)
    g_raw, _, A_log, dt_bias = _raw(inp, 12)
    got = kda_lib.gate_cumsum(g_raw, chunk_size=chunk, g_scale=RCP_LN2, A_log=A_log,
                              dt_bias=dt_bias)
    import oracle

    want = oracle.gate_cumsum(oact.gate(g_raw, A_log, dt_bias), chunk=chunk, g_scale=RCP_LN2)
    err = np.max(np.abs(got.cpu().double().numpy() - want)) / np.max(np.abs(want))
    assert err <= 1e-5, err
