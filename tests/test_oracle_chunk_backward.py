"""Pins of the chunk-form backward oracle (CPU): every gradient against the
reverse-mode derivative of the token recurrence (oracle/backward.py, an independent
derivation), the reverse scan's per-chunk state gradients against the recurrence's
own gradients of its states at the chunk boundaries, and planted mistakes that the
first pin must catch."""
import math

import numpy as np
import pytest

from oracle import backward as ob
from oracle import chunk_backward as cb

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def _problem(seed, B=1, T=11, H=1, HV=2, K=3, V=2, lens=(4, 0, 7), h0=True):
    r = np.random.default_rng(seed)
    p = dict(q=r.standard_normal((B, T, H, K)), k=0.6 * r.standard_normal((B, T, H, K)),
             v=r.standard_normal((B, T, HV, V)), g=-r.uniform(0.05, 0.6, (B, T, HV, K)),
             beta=r.uniform(0.2, 0.9, (B, T, HV)), do=r.standard_normal((B, T, HV, V)))
    p["cu"] = None if lens is None else np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = B if lens is None else len(lens)
    p["h0"] = 0.3 * r.standard_normal((N, HV, K, V)) if h0 else None
    p["dht"] = r.standard_normal((N, HV, K, V)) if h0 else None
    return p


def _both(p, chunk_size, g_scale=1.0):
    args = (p["q"], p["k"], p["v"], p["g"], p["beta"], p["do"], p["h0"], p["dht"])
    ref = ob.recurrent_grads(*args, cu_seqlens=p["cu"], g_scale=g_scale)
    got = cb.chunk_grads(*args, cu_seqlens=p["cu"], g_scale=g_scale, chunk_size=chunk_size)
    return got, ref


def _err(got, ref):
    return {n: float(np.abs(got[n] - ref[n]).max() / max(1e-300, np.abs(ref[n]).max()))
            for n in NAMES if ref[n] is not None}


@pytest.mark.parametrize("chunk_size", [1, 3, 4, 64])
def test_packed_with_empty_slot_and_partial_chunks(chunk_size):
    got, ref = _both(_problem(1), chunk_size)
    assert max(_err(got, ref).values()) < 1e-12, _err(got, ref)


def test_dense_grouped_heads_natural_log_gate():
    p = _problem(2, B=2, T=9, H=2, HV=4, K=4, V=3, lens=None)
    got, ref = _both(p, 4, g_scale=1.0 / math.log(2.0))
    assert max(_err(got, ref).values()) < 1e-12, _err(got, ref)


def test_without_initial_state_or_final_gradient():
    got, ref = _both(_problem(3, lens=(11,), h0=False), 4)
    assert got["dh0"] is None
    assert max(_err(got, ref).values()) < 1e-12, _err(got, ref)


def test_reverse_scan_state_gradients_match_the_recurrence():
    """Stage 4's dL/dh at every chunk boundary equals the gradient of the loss with
    respect to the recurrence's state there (torch reverse mode on the recurrence), the
    state taken as a copy that only the tokens after the boundary (and dht) read: the
    boundary token's own readout is part of its chunk."""
    import torch

    p = _problem(4, lens=None, T=10, HV=1, K=3, V=2)
    cs = 4
    got = cb.chunk_grads(p["q"], p["k"], p["v"], p["g"], p["beta"], p["do"], p["h0"], p["dht"],
                         chunk_size=cs, stages=True)
    q, k, v, g, beta, do = (torch.tensor(p[x]) for x in ("q", "k", "v", "g", "beta", "do"))
    S = torch.tensor(p["h0"][0, 0], requires_grad=True)
    scale = 1.0 / math.sqrt(3)
    states, loss = [], torch.zeros((), dtype=torch.float64)
    for t in range(10):
        S = torch.exp2(g[0, t, 0])[:, None] * S
        delta = beta[0, t, 0] * (v[0, t, 0] - S.T @ k[0, t, 0])
        S = S + torch.outer(k[0, t, 0], delta)
        loss = loss + (scale * (S.T @ q[0, t, 0]) * do[0, t, 0]).sum()
        if (t + 1) % cs == 0 or t == 9:
            S = S.clone()
            S.retain_grad()
            states.append(S)
    loss = loss + (S * torch.tensor(p["dht"][0, 0])).sum()
    loss.backward()
    chunks = got["chunks"][(0, 0)]
    assert len(chunks) == len(states) == 3
    for c, st in enumerate(states):
        assert np.allclose(chunks[c]["dh_next"], st.grad.numpy(), rtol=1e-12, atol=1e-12), c


@pytest.mark.parametrize("mutant", ["forward_cumsum", "no_ln2"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "forward_cumsum":
        monkeypatch.setattr(cb, "_reverse_cumsum", lambda x: np.cumsum(x, axis=0))
    else:
        monkeypatch.setattr(cb, "LN2", 1.0)
    got, ref = _both(_problem(5), 4)
    assert _err(got, ref)["dg"] > 1e-3


def test_l2norm_option():
    p = _problem(6)
    p["q"] *= 2.5
    args = (p["q"], p["k"], p["v"], p["g"], p["beta"], p["do"], p["h0"], p["dht"])
    ref = ob.recurrent_grads(*args, cu_seqlens=p["cu"], l2norm=True)
    got = cb.chunk_grads(*args, cu_seqlens=p["cu"], chunk_size=4, l2norm=True)
    assert max(_err(got, ref).values()) < 1e-12, _err(got, ref)


@pytest.mark.parametrize("bias,beta_scale", [(True, 2.0), (False, 0.0)])
def test_activation_options(bias, beta_scale):
    p = _problem(7)
    r = np.random.default_rng(8)
    g_raw = r.standard_normal(p["g"].shape) - 1.0
    b_raw = r.standard_normal(p["beta"].shape) if beta_scale else p["beta"]
    A_log = r.uniform(-0.5, 0.8, 2)
    dt_bias = 0.5 * r.standard_normal((2, 3)) if bias else None
    args = (p["q"], p["k"], p["v"], g_raw, b_raw, p["do"], p["h0"], p["dht"])
    kw = dict(cu_seqlens=p["cu"], g_scale=1.0 / math.log(2.0), A_log=A_log, dt_bias=dt_bias,
              beta_scale=beta_scale)
    ref = ob.recurrent_grads(*args, **kw)
    got = cb.chunk_grads(*args, chunk_size=4, **kw)
    names = NAMES + ("dA_log",) + (("ddt_bias",) if bias else ())
    err = {n: float(np.abs(got[n] - ref[n]).max() / np.abs(ref[n]).max()) for n in names}
    assert max(err.values()) < 1e-12, err
    if not bias:
        assert got["ddt_bias"] is None


def test_options_ignore_rows_past_the_last_offset():
    """NaN in every input row past the last offset changes no gradient (the rows belong
    to no sequence), with the norm and both activations on."""
    p = _problem(9, T=14)
    r = np.random.default_rng(10)
    g_raw = r.standard_normal(p["g"].shape) - 1.0
    b_raw = r.standard_normal(p["beta"].shape)
    for x in (p["q"], p["k"], g_raw, b_raw):
        x[:, 11:] = np.nan
    args = (p["q"], p["k"], p["v"], g_raw, b_raw, p["do"], p["h0"], p["dht"])
    kw = dict(cu_seqlens=p["cu"], g_scale=1.0 / math.log(2.0), l2norm=True,
              A_log=r.uniform(-0.5, 0.8, 2), dt_bias=0.5 * r.standard_normal((2, 3)),
              beta_scale=1.0)
    ref = ob.recurrent_grads(*args, **kw)
    got = cb.chunk_grads(*args, chunk_size=4, **kw)
    names = NAMES + ("dA_log", "ddt_bias")
    err = {n: float(np.abs(got[n][:, :11] - ref[n][:, :11]).max() / np.abs(ref[n]).max())
           if n not in ("dh0", "dA_log", "ddt_bias") else
           float(np.abs(got[n] - ref[n]).max() / np.abs(ref[n]).max()) for n in names}
    assert max(err.values()) < 1e-12, err
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.all(got[n][:, 11:] == 0), n
