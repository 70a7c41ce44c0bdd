"""GPU unit test of the tcgen05/TMA/TMEM building blocks (csrc/tc.cuh): a 128 x N x 128
bf16 GEMM with each operand layout the kernels use, against torch in fp32."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from gated_delta_rule_16_gb300 import build
    out = os.path.join(HERE, "_build", "libtcunit.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    src = os.path.join(HERE, "csrc", "tc_unit.cu")
    subprocess.check_call([build.nvcc(), *build.ARCH, "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                           src, "-o", out])
    l = ctypes.CDLL(out)
    l.tc_gemm.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
    l.tc_gemm.restype = ctypes.c_int
    return l


@pytest.mark.parametrize("N", [64, 128, 256])
@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("a_manual", [0, 1])
def test_tc_gemm(lib, N, b_mn, a_manual):
    torch.manual_seed(N + 10 * b_mn + 100 * a_manual)
    dev = torch.device("cuda:0")
    A = torch.randn(128, 128, device=dev).bfloat16()
    Bkn = torch.randn(128, N, device=dev).bfloat16()          # [K][N]
    B = Bkn.contiguous() if b_mn else Bkn.t().contiguous()    # MN-major [K][N] or K-major [N][K]
    Af = A.float().contiguous()
    D = torch.full((128, N), float("nan"), device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.tc_gemm(A.data_ptr(), Af.data_ptr(), B.data_ptr(), b_mn, a_manual, N, D.data_ptr(), err.data_ptr())
    assert rc == 0 and err.item() == 0, (rc, err.item())
    ref = A.float() @ Bkn.float()
    assert torch.isfinite(D).all()
    assert (D - ref).abs().max().item() <= 1e-3 * ref.abs().max().item()
