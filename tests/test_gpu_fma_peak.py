"""The fp32 FMA peak microbenchmark (the denominator of the fp32-bound rooflines)
returns a plausible figure: within a factor of two of SMs x 128 lanes x 2 flops
x the maximum SM clock."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_fma_peak_is_plausible(kda_lib):
    dev = torch.cuda.current_device()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nominal = sms * 128 * 2 * 2.07e9 / 1e12  # TFLOP/s at 2070 MHz
    peak = kda_lib.kda_measure_fp32_fma_peak()
    assert 0.5 * nominal <= peak <= 1.2 * nominal, (peak, nominal)
