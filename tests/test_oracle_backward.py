"""Pins of the backward oracle (CPU): its gradients against central finite
differences of the C oracle's forward (a separate implementation of the
recurrence), against the closed form at beta = 0, and a planted mistake that the
finite differences must catch."""
import math

import numpy as np
import pytest

import oracle
from oracle import backward as ob


def _problem(seed, B=1, T=5, H=1, HV=2, K=3, V=2, packed=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, H, K))
    k = r.standard_normal((B, T, H, K)) * 0.6
    v = r.standard_normal((B, T, HV, V))
    g = -r.uniform(0.05, 0.6, (B, T, HV, K))
    beta = r.uniform(0.2, 0.9, (B, T, HV))
    cu = np.array([0, 2, 2, 5], dtype=np.int32) if packed else None
    N = 3 if packed else B
    h0 = 0.3 * r.standard_normal((N, HV, K, V))
    do = r.standard_normal((B, T, HV, V))
    dht = r.standard_normal((N, HV, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, do=do, dht=dht, cu=cu)


def _loss(p, g_scale=1.0, l2norm=False):
    """sum(o * do) + sum(ht * dht) through the C oracle's forward."""
    o, ht = oracle.recurrent(p["q"], p["k"], p["v"], p["g"], p["beta"], h0=p["h0"],
                             cu_seqlens=p["cu"], g_scale=g_scale, l2norm=l2norm, o_fill=0.0)
    return float((o * p["do"]).sum() + (ht * p["dht"]).sum())


def _fd(p, name, g_scale=1.0, eps=1e-6, l2norm=False):
    x = p[name]
    out = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        keep = x[idx]
        x[idx] = keep + eps
        up = _loss(p, g_scale, l2norm)
        x[idx] = keep - eps
        dn = _loss(p, g_scale, l2norm)
        x[idx] = keep
        out[idx] = (up - dn) / (2 * eps)
    return out


@pytest.mark.parametrize("packed,g_scale", [(True, 1.0), (False, 1.0 / math.log(2.0))])
def test_gradients_match_finite_differences_of_the_c_oracle(packed, g_scale):
    p = _problem(3 if packed else 4, B=1 if packed else 2, packed=packed)
    got = ob.recurrent_grads(p["q"], p["k"], p["v"], p["g"], p["beta"], p["do"], p["h0"],
                             p["dht"], cu_seqlens=p["cu"], g_scale=g_scale)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                      ("h0", "dh0")):
        want = _fd(p, name, g_scale)
        err = np.abs(got[key] - want).max() / max(1e-12, np.abs(want).max())
        assert err < 1e-6, (name, err)


def test_empty_slot_passes_the_state_gradient_through():
    p = _problem(5)
    got = ob.recurrent_grads(p["q"], p["k"], p["v"], p["g"], p["beta"], p["do"], p["h0"],
                             p["dht"], cu_seqlens=p["cu"])
    assert np.array_equal(got["dh0"][1], p["dht"][1])  # slot 1 is empty


def test_closed_form_at_beta_zero():
    """beta = 0: S_t = D_t h0 with D_t = 2^(cumsum g), so o_t = scale (D_t h0)^T q_t:
    dq_t = scale (D_t h0) do_t, dk = dv = 0, dh0 = sum_t scale D_t q_t do_t^T + D_T dht."""
    p = _problem(6, B=1, T=4, H=1, HV=1, K=3, V=2, packed=False)
    p["beta"][:] = 0.0
    got = ob.recurrent_grads(p["q"], p["k"], p["v"], p["g"], p["beta"], p["do"], p["h0"],
                             p["dht"])
    scale = 1.0 / math.sqrt(3)
    D = np.exp2(np.cumsum(p["g"][0, :, 0], axis=0))  # [T, K]
    h0 = p["h0"][0, 0]
    dq = np.stack([scale * (D[t][:, None] * h0) @ p["do"][0, t, 0] for t in range(4)])
    assert np.allclose(got["dq"][0, :, 0], dq, atol=1e-12)
    assert np.allclose(got["dk"], 0, atol=1e-12) and np.allclose(got["dv"], 0, atol=1e-12)
    dh0 = sum(scale * D[t][:, None] * np.outer(p["q"][0, t, 0], p["do"][0, t, 0]) for t in range(4))
    dh0 = dh0 + D[3][:, None] * p["dht"][0, 0]
    assert np.allclose(got["dh0"][0, 0], dh0, atol=1e-12)


def test_a_planted_sign_error_fails_the_finite_differences():
    """The finite-difference pin discriminates: the gradients of a recurrence with
    the residual's sign flipped (delta = beta (v + S^T k)) are far from it."""
    import torch

    p = _problem(7, packed=False)
    want = _fd(p, "k")
    kk = torch.tensor(p["k"], requires_grad=True)
    q, v, g, beta = (torch.tensor(p[x]) for x in ("q", "v", "g", "beta"))
    S = torch.tensor(p["h0"][0])
    loss = torch.zeros((), dtype=torch.float64)
    for t in range(p["q"].shape[1]):
        kt = kk[0, t].repeat_interleave(2, 0)
        qt = q[0, t].repeat_interleave(2, 0)
        S = torch.exp2(g[0, t])[:, :, None] * S
        delta = beta[0, t][:, None] * (v[0, t] + torch.einsum("hkv,hk->hv", S, kt))  # planted
        S = S + kt[:, :, None] * delta[:, None, :]
        loss = loss + (torch.einsum("hkv,hk->hv", S, qt) / math.sqrt(3) * torch.tensor(p["do"][0, t])).sum()
    loss = loss + (S * torch.tensor(p["dht"][0])).sum()
    loss.backward()
    err = np.abs(kk.grad.numpy() - want).max() / np.abs(want).max()
    assert err > 1e-2


def test_l2norm_gradients_match_finite_differences():
    p = _problem(8)
    p["q"] *= 2.5  # unnormalised rows
    got = ob.recurrent_grads(p["q"], p["k"], p["v"], p["g"], p["beta"], p["do"], p["h0"],
                             p["dht"], cu_seqlens=p["cu"], l2norm=True)
    for name, key in (("q", "dq"), ("k", "dk"), ("g", "dg"), ("beta", "dbeta")):
        want = _fd(p, name, l2norm=True)
        err = np.abs(got[key] - want).max() / max(1e-12, np.abs(want).max())
        assert err < 1e-6, (name, err)
    # a row's gradient is orthogonal to the row itself up to the epsilon: rescaling q
    # leaves the output unchanged
    dots = (got["dq"] * p["q"]).sum(-1)
    assert np.abs(dots).max() < 1e-5 * np.abs(got["dq"]).max() * np.abs(p["q"]).max()


def test_activation_gradients_match_finite_differences():
    """Raw gate through -exp(A_log) softplus(g + dt_bias) and raw beta through
    sigmoid * 2 (fp32 values: no rounding), against finite differences of the C
    recurrence fed by the oracle's own activations."""
    from oracle import activation as act

    p = _problem(9)
    r = np.random.default_rng(10)
    p["graw"] = r.standard_normal(p["g"].shape) - 1.0
    p["braw"] = r.standard_normal(p["beta"].shape)
    p["A_log"] = r.uniform(-0.5, 0.8, 2)
    p["dt_bias"] = 0.5 * r.standard_normal((2, 3))
    gs = 1.0 / math.log(2.0)

    def loss(pp):
        o, ht = oracle.recurrent(pp["q"], pp["k"], pp["v"],
                                 act.gate(pp["graw"], pp["A_log"], pp["dt_bias"]),
                                 act.beta(pp["braw"], 2.0), h0=pp["h0"], cu_seqlens=pp["cu"],
                                 g_scale=gs, o_fill=0.0)
        return float((o * pp["do"]).sum() + (ht * pp["dht"]).sum())

    got = ob.recurrent_grads(p["q"], p["k"], p["v"], p["graw"], p["braw"], p["do"], p["h0"],
                             p["dht"], cu_seqlens=p["cu"], g_scale=gs, A_log=p["A_log"],
                             dt_bias=p["dt_bias"], beta_scale=2.0)
    for name, key in (("graw", "dg"), ("braw", "dbeta"), ("A_log", "dA_log"),
                      ("dt_bias", "ddt_bias"), ("k", "dk")):
        x = p[name]
        want = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            keep = x[idx]
            x[idx] = keep + 1e-6
            up = loss(p)
            x[idx] = keep - 1e-6
            dn = loss(p)
            x[idx] = keep
            want[idx] = (up - dn) / 2e-6
        err = np.abs(got[key] - want).max() / max(1e-12, np.abs(want).max())
        assert err < 1e-6, (name, err)
