import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def kda_lib():
    """The CUDA library through its Python binding; the GPU tests need it loaded."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_cumsum_gb300 as kda

    kda.load()  # raises if the extension is missing: there is no fallback
    return kda
