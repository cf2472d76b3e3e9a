"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_recurrence_pin(check):
    check(oracle.recurrent)


@pytest.mark.parametrize("check", oracle_pins.CUMSUM_CHECKS, ids=lambda c: c.__name__)
def test_gate_cumsum_pin(check):
    check(oracle.gate_cumsum)


def test_oracle_rejects_bad_offsets():
    g = np.zeros((1, 8, 1, 1))
    for cu in ([1, 4, 8], [0, 5, 4], [0, 4, 9]):
        with pytest.raises(ValueError):
            oracle.gate_cumsum(g, cu_seqlens=np.array(cu, dtype=np.int32))


def test_oracle_bf16_inputs_upcast_exactly():
    """The oracle sees the exact values of low-precision inputs."""
    import torch

    x = torch.randn(1, 5, 1, 8).to(torch.bfloat16)
    from oracle import _f64

    assert np.array_equal(_f64(x), x.float().double().numpy())
