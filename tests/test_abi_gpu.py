"""The C ABI on a GPU: every rejected call returns its code and writes nothing."""
import ctypes

import pytest
import torch

import exact_attention_32_gb300 as fa

pytestmark = pytest.mark.gpu


def raw(q, k, v, o, lse, B, H, N, d, scale=0.125, causal=0):
    return fa.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, 0)


@pytest.fixture
def bufs():
    B, H, N, d = 1, 2, 256, 64
    q = torch.randn(B, H, N, d, device="cuda").bfloat16()
    o = torch.full_like(q, 7.0)
    lse = torch.full((B, H, N), 7.0, device="cuda")
    return q, o, lse, (B, H, N, d)


def untouched(o, lse):
    torch.cuda.synchronize()
    return bool((o == 7.0).all()) and bool((lse == 7.0).all())


def test_device_is_sm103():
    assert torch.cuda.get_device_capability() == (10, 3)


def test_valid_call_returns_ok(bufs):
    q, o, lse, (B, H, N, d) = bufs
    assert raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d) == 0
    assert fa.fa_get_device_status(0) == 0
    assert not untouched(o, lse)


def test_misaligned_pointer(bufs):
    q, o, lse, (B, H, N, d) = bufs
    assert raw(q.data_ptr() + 2, q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d) == 1
    assert untouched(o, lse)


def test_lse_needs_only_four_byte_alignment(bufs):
    q, o, lse, (B, H, N, d) = bufs
    big = torch.full((B * H * N + 4,), 7.0, device="cuda")
    assert raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), big.data_ptr() + 2, B, H, N, d) == 1
    assert untouched(o, lse)
    assert raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), big.data_ptr() + 4, B, H, N, d) == 0
    torch.cuda.synchronize()
    assert bool((big[0] == 7.0)) and bool(torch.isfinite(big[1:1 + B * H * N]).all()) and bool((big[-3:] == 7.0).all())


def test_null_pointer(bufs):
    q, o, lse, (B, H, N, d) = bufs
    assert raw(0, q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d) == 1
    assert untouched(o, lse)


def test_host_pointer(bufs):
    q, o, lse, (B, H, N, d) = bufs
    host = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
    assert raw(host.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d) == 1
    assert untouched(o, lse)


def test_output_overlapping_input(bufs):
    q, o, lse, (B, H, N, d) = bufs
    assert raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), lse.data_ptr(), B, H, N, d) == 1
    assert raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), o.data_ptr(), B, H, N, d) == 1
    assert untouched(o, lse)


def test_unsupported_head_dim(bufs):
    q, o, lse, (B, H, N, d) = bufs
    assert raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N // 2, 128) == 0
    assert raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, 96) == 2


def test_forward_argument_checks():
    q = torch.randn(1, 1, 64, 64, device="cuda").bfloat16()
    with pytest.raises(ValueError):
        fa.forward(q.float(), q, q)
    with pytest.raises(ValueError):
        fa.forward(q, q[:, :, :32], q)
    with pytest.raises(fa.FAError) as e:
        fa.forward(q, q, q, scale=-1.0)
    assert e.value.status == 1
