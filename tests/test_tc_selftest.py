"""Device building blocks of the attention kernel.

tcgen05 operand layouts the attention kernel relies on, checked bit-exactly
on small-integer data (every product and sum is exact in fp32):
S = Q K^T with both operands K-major and 128-byte swizzled in shared memory,
then P = bf16(S) written into tensor memory over S, and O = P V with P read
from tensor memory and V an MN-major shared-memory operand."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from exact_attention_32_gb300 import build as fa_build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def selftest_lib():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libtcselftest.so")
    subprocess.run([fa_build.nvcc()] + fa_build.ARCH +
                   ["-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", fa_build.CSRC,
                    os.path.join(HERE, "cuda", "tc_selftest.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.tc_selftest.restype = ctypes.c_int
    lib.tc_selftest.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int]
    lib.wait_timeout_selftest.restype = ctypes.c_int
    lib.wait_timeout_selftest.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]
    return lib


@pytest.mark.parametrize("d", [64, 128])
def test_mma_layouts_bit_exact(selftest_lib, d):
    g = torch.Generator().manual_seed(d)
    q = torch.randint(-2, 3, (128, d), generator=g).to(torch.bfloat16)
    k = torch.randint(-2, 3, (128, d), generator=g).to(torch.bfloat16)
    v = torch.randint(-2, 3, (128, d), generator=g).to(torch.bfloat16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    s_out = torch.full((128, 128), float("nan"), device="cuda")
    o_out = torch.full((128, d), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = selftest_lib.tc_selftest(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), s_out.data_ptr(),
                                  o_out.data_ptr(), status.data_ptr(), d)
    assert rc == 0
    assert int(status.item()) == 0
    s_ref = q.double() @ k.double().T
    assert torch.equal(s_out.cpu().double(), s_ref), "S = Q K^T layout mismatch"
    p = s_ref.float().to(torch.bfloat16).double()
    o_ref = p @ v.double()
    assert torch.equal(o_out.cpu().double(), o_ref), "O = P V layout mismatch"


def test_bounded_wait_gives_up_and_context_survives(selftest_lib):
    # the same bounded mbarrier wait every pipeline stage of the kernel uses:
    # nothing arrives, so it must return "timed out" after about its limit,
    # and the CUDA context must stay usable afterwards
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit_ns = 50_000_000
    rc = selftest_lib.wait_timeout_selftest(status.data_ptr(), limit_ns, elapsed.data_ptr())
    assert rc == 0
    assert status.tolist() == [1, 1]  # timed out; the previous-phase wait passed at once
    assert limit_ns <= int(elapsed.item()) < 20 * limit_ns
    x = torch.arange(1000, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 499500.0


def test_tensor_memory_load_with_max(selftest_lib):
    # the reducing tensor-memory load returns the values unchanged and, per
    # thread, the largest of the 32 it loaded; rows hold negative values,
    # -inf (masked keys), all--inf pieces and ties
    selftest_lib.ld_max_selftest.restype = ctypes.c_int
    selftest_lib.ld_max_selftest.argtypes = [ctypes.c_void_p] * 3
    g = torch.Generator().manual_seed(7)
    x = torch.randn((128, 128), generator=g) * 30
    x[::3, 5::7] = float("-inf")
    x[5, 32:64] = float("-inf")
    x[9, :] = -1.0
    x[11, 70] = 1e30
    x[12, 96:128] = -3.5
    xd = x.cuda()
    vals = torch.empty_like(xd)
    mx = torch.empty((128, 4), device="cuda")
    assert selftest_lib.ld_max_selftest(xd.data_ptr(), vals.data_ptr(), mx.data_ptr()) == 0
    assert torch.equal(vals.cpu(), x)
    assert torch.equal(mx.cpu(), x.view(128, 4, 32).amax(dim=2))
