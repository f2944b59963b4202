"""fa_fwd_splitkv_noalloc: the split-KV forward for callers that cannot
allocate device memory (engines that plan all device memory at start-up,
plugins handed only their input and output tensors, loops that cannot afford
a cudaMalloc).  Its scratch is a static device array inside the library.

Called through the C ABI (ctypes on libfa.so) twice in a row, on different
inputs so that the second call runs over the first call's leftovers in the
shared array, and each result is compared with fa_fwd_splitkv given a
caller-allocated workspace.  Both run the same kernels on the same data with
only the scratch address differing, so the outputs must be bit-identical (a
part left stale from the first call would show).  This file is collected last
so that a run stopping at the first failure has run every other test first; it
also passes on its own in a fresh process.  The argument checks, which make no
CUDA call, are compared with fa_fwd_splitkv's on the CPU.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_32_gb300 import build as fa_build
from exact_attention_32_gb300 import make_inputs

MAX_O, MEAN_O, MAX_LSE = 2e-2, 2e-3, 1e-3
LIMIT = 32 * 1024 * 1024  # FA_SPLITKV_NOALLOC_MAX_BYTES
FA_ERR_WORKSPACE_LIMIT = 7


@pytest.fixture(scope="module")
def lib():
    L = ctypes.CDLL(fa_build.build())
    vp, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
    L.fa_fwd_splitkv_noalloc.restype = ctypes.c_int
    L.fa_fwd_splitkv_noalloc.argtypes = [vp] * 5 + [i64] * 4 + [f32, ctypes.c_int, i64, vp]
    L.fa_fwd_splitkv.restype = ctypes.c_int
    L.fa_fwd_splitkv.argtypes = [vp] * 5 + [i64] * 4 + [f32, ctypes.c_int, i64, vp, i64, vp]
    L.fa_fwd_splitkv_workspace_bytes.restype = i64
    L.fa_fwd_splitkv_workspace_bytes.argtypes = [i64] * 5
    L.fa_status_string.restype = ctypes.c_char_p
    L.fa_status_string.argtypes = [ctypes.c_int]
    L.fa_get_device_status.restype = ctypes.c_int
    L.fa_get_device_status.argtypes = [vp]
    return L


def run(lib, noalloc, q, k, v, scale, causal, S):
    B, H, N, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device=q.device)
    stream = torch.cuda.current_stream().cuda_stream
    if noalloc:
        st = lib.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        B, H, N, d, scale, int(causal), S, stream)
    else:
        need = lib.fa_fwd_splitkv_workspace_bytes(B, H, N, d, S)
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
        st = lib.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, H, N, d, scale, int(causal), S, ws.data_ptr(), need, stream)
    assert st == 0, lib.fa_status_string(st)
    assert lib.fa_get_device_status(None) == 0
    return o.cpu(), lse.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,causal,S", [(2, 4, 1000, 128, True, 3), (1, 8, 700, 64, False, 4)])
def test_noalloc_matches_workspace_version_twice(lib, B, H, N, d, causal, S):
    assert lib.fa_fwd_splitkv_workspace_bytes(B, H, N, d, S) <= LIMIT
    scale = float(np.float32(1 / np.sqrt(d)))
    for call in range(2):
        q, k, v = (t.cuda() for t in make_inputs(B, H, N, d, seed=7000 + 10 * call + d, q_gain=1.0 + 3 * call))
        o1, l1 = run(lib, True, q, k, v, scale, causal, S)
        o2, l2 = run(lib, False, q, k, v, scale, causal, S)
        assert torch.isfinite(o1.float()).all() and torch.isfinite(l1).all()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("B,H,N,d,scale,causal,S", [
    (0, 1, 128, 64, 0.125, 0, 2), (1, 1, 0, 64, 0.125, 0, 2), (1, 1, 128, 96, 0.125, 0, 2),
    (1, 1, (1 << 31) - 100, 256, 0.125, 0, 2), (1 << 20, 1 << 20, 4, 64, 0.125, 0, 2),
    (1, 1, 128, 64, 0.0, 0, 2), (1, 1, 128, 64, float("nan"), 0, 2), (1, 1, 128, 64, 0.125, 2, 2),
    (1, 1, 128, 64, 0.125, 0, 0), (1, 1, 128, 64, 0.125, 0, 33), (1, 2, 128, 96, 0.125, 0, 40)])
def test_argument_errors_match_the_workspace_version(lib, B, H, N, d, scale, causal, S):
    # every case fails the size, scale, causal or n_splits rules, which both
    # entry points check before any CUDA call and in the same order
    args = (None,) * 5 + (B, H, N, d, scale, causal, S)
    a = lib.fa_fwd_splitkv_noalloc(*args, None)
    b = lib.fa_fwd_splitkv(*args, None, 1 << 40, None)
    assert a == b and a != 0, (a, b)


def test_limit_is_checked_before_any_device_call(lib):
    # a valid problem whose parts exceed the array: refused from the sizes alone
    B, H, N, d, S = 1, 32, 4096, 128, 4
    assert lib.fa_fwd_splitkv_workspace_bytes(B, H, N, d, S) > LIMIT
    assert lib.fa_fwd_splitkv_noalloc(*(None,) * 5, B, H, N, d, 0.125, 0, S, None) == FA_ERR_WORKSPACE_LIMIT


@pytest.mark.gpu
def test_noalloc_refuses_problems_beyond_its_array(lib):
    B, H, N, d, S = 1, 32, 4096, 128, 4
    assert lib.fa_fwd_splitkv_workspace_bytes(B, H, N, d, S) > LIMIT
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 7.0)
    lse = torch.full((B, H, N), 7.0, device="cuda")
    st = lib.fa_fwd_splitkv_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    B, H, N, d, 0.125, 0, S, None)
    assert st == FA_ERR_WORKSPACE_LIMIT
    assert lib.fa_status_string(st).decode().startswith("FA_ERR_WORKSPACE_LIMIT")
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
