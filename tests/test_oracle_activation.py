"""Pins of the oracle's input activations (CPU): closed forms the mathematics
fixes, checked so that a plausible mistake in the activation (a dropped term, a
wrong sign, a transposed bias, exp for softplus, a missing scale) fails at least
one of them; each such mistake is planted in a copy below and must be caught."""
import math

import numpy as np
import pytest

from oracle import activation as act

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

HV, K = 3, 5


def _params(seed=0):
    rng = np.random.default_rng(seed)
    A = rng.normal(size=HV)
    bias = rng.normal(size=(HV, K))  # deliberately not symmetric in (hv, d)
    return A, bias


def pin_zero_point(gate_fn):
    """g = -dt_bias puts softplus at its zero point ln 2, so the decay is
    -exp(A_log[hv]) ln 2 for every token and channel of head hv."""
    A, bias = _params()
    g_raw = np.broadcast_to(-bias, (2, 4, HV, K)).copy()
    want = np.broadcast_to((-np.exp(A) * math.log(2.0))[None, None, :, None], g_raw.shape)
    return np.allclose(gate_fn(g_raw, A, bias), want, rtol=1e-14, atol=0)


def pin_asymptotes(gate_fn):
    """softplus(x) -> x for large x and -> e^x for very negative x."""
    A = np.zeros(HV)
    big = np.full((1, 1, HV, K), 40.0)
    small = np.full((1, 1, HV, K), -40.0)
    ok_big = np.allclose(gate_fn(big, A), -40.0 - math.exp(-40.0), rtol=1e-15, atol=0)
    ok_small = np.allclose(gate_fn(small, A), -math.exp(-40.0), rtol=1e-12, atol=0)
    return ok_big and ok_small


def pin_no_bias_is_zero_bias(gate_fn):
    """dt_bias = None and dt_bias = 0 agree, and a bias shifts the argument."""
    A, bias = _params(1)
    g = np.random.default_rng(2).normal(size=(2, 3, HV, K))
    same = np.array_equal(gate_fn(g, A), gate_fn(g, A, np.zeros((HV, K))))
    shifted = np.allclose(gate_fn(g - bias, A, bias), gate_fn(g, A), rtol=1e-14, atol=0)
    return same and shifted


def pin_beta(beta_fn):
    """sigmoid(0) = 1/2, sigmoid(+-ln 3) = 3/4, 1/4; the scale multiplies; bf16
    results lie on the bf16 grid."""
    import torch

    x = np.array([0.0, math.log(3.0), -math.log(3.0), 50.0])
    ok = True
    for s in (1.0, 2.0):
        ok &= np.allclose(beta_fn(x, s), s * np.array([0.5, 0.75, 0.25, 1.0]), rtol=1e-15, atol=0)
    y = beta_fn(np.array([0.1, -0.7, 1.3]), 2.0, bf16=True)
    on_grid = torch.from_numpy(y).to(torch.bfloat16).to(torch.float64).numpy()
    ok &= np.array_equal(y, on_grid)
    ok &= np.allclose(y, 2.0 / (1.0 + np.exp(-np.array([0.1, -0.7, 1.3]))), rtol=2 ** -8, atol=0)
    return bool(ok)


GATE_PINS = [pin_zero_point, pin_asymptotes, pin_no_bias_is_zero_bias]


@pytest.mark.parametrize("pin", GATE_PINS, ids=[p.__name__ for p in GATE_PINS])
def test_gate_pins(pin):
    assert pin(act.gate)


def test_beta_pin():
    assert pin_beta(act.beta)


def _gate_sign(g, A, b=None):
    return -act.gate(g, A, b)


def _gate_exp_for_softplus(g, A, b=None):
    x = g if b is None else g + b[None, None]
    return -np.exp(A)[None, None, :, None] * np.exp(x)


def _gate_bias_transposed(g, A, b=None):
    return act.gate(g, A, None if b is None else np.ascontiguousarray(b[::-1, ::-1]))


def _gate_log_a(g, A, b=None):
    x = g if b is None else g + b[None, None]
    return -A[None, None, :, None] * act.softplus(x)


def _gate_bias_dropped(g, A, b=None):
    return act.gate(g, A, None)


GATE_MUTANTS = [_gate_sign, _gate_exp_for_softplus, _gate_bias_transposed, _gate_log_a,
                _gate_bias_dropped]


@pytest.mark.parametrize("mutant", GATE_MUTANTS, ids=[m.__name__ for m in GATE_MUTANTS])
def test_gate_mutant_is_caught(mutant):
    assert not all(pin(mutant) for pin in GATE_PINS)


def _beta_no_scale(x, s, bf16=False):
    return act.beta(x, 1.0, bf16)


def _beta_tanh(x, s, bf16=False):
    return s * np.tanh(np.asarray(x, dtype=np.float64))


def _beta_not_rounded(x, s, bf16=False):
    return act.beta(x, s, False)


@pytest.mark.parametrize("mutant", [_beta_no_scale, _beta_tanh, _beta_not_rounded],
                         ids=["no_scale", "tanh", "not_rounded"])
def test_beta_mutant_is_caught(mutant):
    assert not pin_beta(mutant)
