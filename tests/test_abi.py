"""The C ABI: the library builds, loads and exports every function include/*.h
declares; host-side validation rejects bad arguments before touching a GPU."""
import ctypes
import glob
import os
import re

import pytest

from exact_attention_32_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        names += re.findall(r"\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libfa():
    path = fa_build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_get_device_status", "fa_status_string", "fa_version"):
        assert n in names


def test_every_declared_symbol_is_exported(libfa):
    for name in declared_functions():
        assert hasattr(libfa, name), name


def test_status_strings(libfa):
    libfa.fa_status_string.restype = ctypes.c_char_p
    for code, tag in enumerate(["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED",
                                "FA_ERR_NO_DEVICE", "FA_ERR_ARCH", "FA_ERR_LAUNCH",
                                "FA_ERR_TIMEOUT"]):
        assert libfa.fa_status_string(code).decode().startswith(tag)
    assert libfa.fa_status_string(99).decode() == "unknown fa_status"
    assert libfa.fa_version() >= 100


def _call(libfa, B=1, H=1, N=128, d=64, scale=0.125, causal=0, ptr=16):
    f = libfa.fa_fwd
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp]
    f.restype = ctypes.c_int
    return f(ptr, ptr, ptr, ptr, ptr, B, H, N, d, scale, causal, None)


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(N=0), dict(N=-5), dict(d=0),
                                dict(scale=0.0), dict(scale=-1.0), dict(scale=float("inf")),
                                dict(scale=float("nan")), dict(causal=2), dict(N=1 << 40)])
def test_invalid_sizes_rejected_before_any_device_call(libfa, kw):
    assert _call(libfa, **kw) == 1  # FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [32, 80, 96, 256])
def test_unsupported_head_dim(libfa, d):
    assert _call(libfa, d=d) == 2  # FA_ERR_UNSUPPORTED


def test_python_binding_exposes_the_abi():
    import exact_attention_32_gb300 as fa
    from exact_attention_32_gb300._binding import EXPORTED
    assert set(EXPORTED) == set(declared_functions())
    for name in EXPORTED:
        assert callable(getattr(fa, name))


def _call_host(libfa, B=1, H=2, N=128, d=64, scale=0.125, causal=0, n_groups=0, ptr=16):
    f = libfa.fa_fwd_host
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [vp] * 10 + [i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, i64, vp]
    f.restype = ctypes.c_int
    return f(*([ptr] * 10), B, H, N, d, scale, causal, n_groups, None)


@pytest.mark.parametrize("kw", [dict(B=0), dict(N=0), dict(scale=0.0), dict(scale=float("nan")), dict(causal=3),
                                dict(n_groups=-1), dict(n_groups=3), dict(B=40, H=2, n_groups=65)])
def test_host_entry_rejects_bad_arguments_before_any_device_call(libfa, kw):
    # n_groups must lie in [1, min(B*H, 64)] (0 = default); B*H = 2 unless given
    assert _call_host(libfa, **kw) == 1  # FA_ERR_INVALID_ARG


def test_host_entry_unsupported_head_dim(libfa):
    assert _call_host(libfa, d=96) == 2  # FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("N,d,causal,expected", [
    (256, 64, 0, "fa_fwd_dp_kernel"), (1000, 64, 1, "fa_fwd_dp_kernel"), (1000, 64, 0, "fa_fwd_dp_kernel"),
    (2048, 64, 1, "fa_fwd_dp_kernel"), (2048, 64, 0, "fa_fwd_tc_kernel"), (4096, 64, 1, "fa_fwd_tc_kernel"),
    (16384, 64, 1, "fa_fwd_tc_kernel"), (256, 128, 0, "fa_fwd_tc_kernel"), (16384, 128, 1, "fa_fwd_tc_kernel")])
def test_forward_kernel_choice(N, d, causal, expected):
    # d = 64 problems whose 256-row units see at most 9 key tiles of 128 on
    # average run on the kernel with P apart from S; all others on the main one
    import exact_attention_32_gb300 as fa
    assert fa.fa_fwd_kernel(2, 3, N, d, causal) == expected
    n_t, n_mb = -(-N // 128), -(-N // 256)
    tiles = sum(min(n_t, 2 * (mb + 1)) if causal else n_t for mb in range(n_mb))
    assert (expected == "fa_fwd_dp_kernel") == (d == 64 and tiles <= 9 * n_mb)


def test_forward_kernel_choice_rejects_bad_arguments(libfa):
    f = libfa.fa_fwd_kernel
    i64 = ctypes.c_int64
    f.argtypes = [i64, i64, i64, i64, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    f.restype = ctypes.c_int
    out = ctypes.c_int(-7)
    assert f(1, 1, 0, 64, 0, ctypes.byref(out)) == 1 and out.value == -7
    assert f(1, 1, 128, 96, 0, ctypes.byref(out)) == 2 and out.value == -7
    assert f(1, 1, 128, 64, 2, ctypes.byref(out)) == 1 and out.value == -7
    assert f(1, 1, 128, 64, 0, None) == 1
