"""Host-side checks of the Python binding (no GPU): tensors that are not on one CUDA
device, or that require grad outside kda_autograd, are rejected before any pointer
reaches the library."""
import pytest
import torch

import gated_delta_rule_cumsum_gb300 as kda


def _cpu_inputs(B=1, T=8, H=1, HV=1, K=8, V=8):
    q = torch.randn(B, T, H, K)
    return dict(q=q, k=torch.randn(B, T, H, K), v=torch.randn(B, T, HV, V),
                g=-torch.rand(B, T, HV, K), beta=torch.rand(B, T, HV))


@pytest.mark.parametrize("fn", ["chunk_kda", "recurrent_kda"])
def test_forward_rejects_host_tensors(fn):
    x = _cpu_inputs()
    with pytest.raises(kda.KdaError) as err:
        getattr(kda, fn)(x["q"], x["k"], x["v"], x["g"], x["beta"])
    assert err.value.status == kda.KDA_ERR_INVALID_ARG


def test_backward_and_autograd_reject_host_tensors():
    x = _cpu_inputs()
    with pytest.raises(kda.KdaError):
        kda.recurrent_kda_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], torch.zeros_like(x["v"]))
    with pytest.raises(kda.KdaError):
        kda.kda_autograd(x["q"], x["k"], x["v"], x["g"], x["beta"])
    with pytest.raises(kda.KdaError):
        kda.gate_cumsum(x["g"])


def test_inputs_requiring_grad_point_to_autograd():
    x = _cpu_inputs()
    x["q"].requires_grad_(True)
    with pytest.raises(kda.KdaError) as err:
        kda.chunk_kda(x["q"], x["k"], x["v"], x["g"], x["beta"])
    assert err.value.status == kda.KDA_ERR_UNSUPPORTED
    assert "kda_autograd" in str(err.value)


def test_activation_parameters_must_be_device_tensors():
    """A host A_log or dt_bias would reach the kernels as a host pointer."""
    with pytest.raises(kda.KdaError):
        kda.make_activation(A_log=torch.zeros(2))
    with pytest.raises(kda.KdaError):
        kda.make_activation(dt_bias=torch.zeros(2, 8))
    act = kda.make_activation(beta_scale=2.0)  # no tensors: nothing to check
    assert act.A_log is None and act.beta_scale == 2.0


def test_one_device_check():
    assert kda._one_device(None, None) is None
    with pytest.raises(kda.KdaError):
        kda._one_device(torch.zeros(1))
    meta = torch.empty(1, device="meta")
    with pytest.raises(kda.KdaError):
        kda._one_device(meta)
