"""The tensor-core building blocks (operand tile layout, shared-memory
descriptors, instruction descriptor, TMEM read-back) on one tile, against a
plain fp32 matmul of the same bf16 values (GPU)."""
import ctypes
import os
import subprocess
import tempfile

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "csrc", "tc_probe.cu")
CSRC = os.path.join(ROOT, "gated_delta_rule_cumsum_gb300", "csrc")


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tmp = tempfile.mkdtemp()
    so = os.path.join(tmp, "tc_probe.so")
    subprocess.run(["nvcc", "-O2", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared", "-I", CSRC, SRC,
                    "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.tc_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
    return lib


@pytest.mark.parametrize("mode", [0, 1, 2, 3], ids=["Ak_Bk", "Ak_Bmn", "Amn_Bk", "Amn_Bmn"])
@pytest.mark.parametrize("N,Kd", [(16, 16), (32, 64), (64, 128), (128, 128), (256, 64)])
def test_single_tile_gemm(probe, mode, N, Kd):
    g = torch.Generator(device="cuda").manual_seed(N * 1000 + Kd + mode)
    A = torch.randn(128, Kd, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(Kd, N, device="cuda", generator=g).to(torch.bfloat16)
    D = torch.full((128, N), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, Kd, mode, err.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(err) == 0
    want = A.float() @ B.float()
    assert torch.allclose(D, want, rtol=1e-4, atol=1e-3), (D - want).abs().max()


# The 128-byte swizzled layouts a TMA copy writes: K-major A and B (the prep's
# gram operands), and a no-swizzle A with an MN-major swizzled B (its W product).
@pytest.mark.parametrize("mode", [4, 8 | 1, 8 | 4 | 1], ids=["Aksw_Bksw", "Ak_Bmnsw", "Aksw_Bmnsw"])
@pytest.mark.parametrize("N,Kd", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_single_tile_gemm_swizzled(probe, mode, N, Kd):
    test_single_tile_gemm(probe, mode, N, Kd)



def test_tmem_16x32bx2_readback(probe):
    """The 16-lane TMEM load with a column offset: thread t < 16 of warp w gets lane
    32 w + t, columns 0..15; thread t >= 16 the same lane 32 w + t - 16, columns
    32..47 -- the layout the backward's M = 64 epilogues read their rows with."""
    probe.tmem_ld16x2_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    out = torch.full((4, 32, 16), float("nan"), device="cuda")
    assert probe.tmem_ld16x2_probe(out.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    w = torch.arange(4, device="cuda").view(4, 1, 1)
    t = torch.arange(32, device="cuda").view(1, 32, 1)
    j = torch.arange(16, device="cuda").view(1, 1, 16)
    want = (32 * w + (t % 16)) * 1000 + j + 32 * (t // 16)
    assert torch.equal(out, want.float())
