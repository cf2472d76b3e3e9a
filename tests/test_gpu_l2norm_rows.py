"""The in-op q/k L2 norm on zero rows and on rows scaled from 1e-3 to 1e3
(attention-gym PR #345, the deferred-norm cases), chunked and recurrent, fp32 and bf16,
against the fp64 oracle applying the same norm (x / sqrt(sum x^2 + 1e-6)) (GPU)."""
import pytest
import torch

from tests.test_gpu_chunk import _check
from tests.test_gpu_chunk import _run as run_chunk
from tests.test_gpu_recurrent import _run as run_recurrent
from tests.test_gpu_recurrent import _small

pytestmark = pytest.mark.gpu


def _extreme_rows(inp, seed):
    gen = torch.Generator().manual_seed(seed)
    for name in ("q", "k"):
        x = inp[name].float().cpu()
        B, T, H, _ = x.shape
        x = x * 10.0 ** (6.0 * torch.rand(B, T, H, 1, generator=gen) - 3.0)
        x[:, ::7] = 0.0
        inp[name] = x.to(inp[name].dtype).cuda()
    return inp


@pytest.mark.parametrize("form", ["chunk", "recurrent"])
@pytest.mark.parametrize("dtype,tol", [(torch.float32, 1e-4), (torch.bfloat16, 2e-2)])
def test_zero_and_extreme_rows(kda_lib, form, dtype, tol):
    inp = _extreme_rows(_small(201, T=90, dtype=dtype), 202)
    run = run_chunk if form == "chunk" else run_recurrent
    o, ht = run(kda_lib, inp, use_qk_l2norm_in_kernel=True)
    assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
    _check(inp, o, ht, tol, l2norm=True)
