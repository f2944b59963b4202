"""fa_fwd_host: the forward on host buffers with the copies pipelined over
groups of (b, h) slices.

GPU: results against the fp64 oracle for ragged groupings (pinned and
pageable host memory); bit-identical to fa_fwd on device-resident inputs (the
same kernel sees the same slices); two calls queued back to back on one
stream reusing the staging buffers; device pointers refused where host
buffers are expected.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import exact_attention_32_gb300 as fa
from exact_attention_32_gb300 import WORKLOADS, make_inputs, workload_inputs
from exact_attention_32_gb300.workloads import sample_rows

MAX_O, MEAN_O, MAX_LSE = 2e-2, 2e-3, 1e-3


def check(o, lse, o_ref, lse_ref):
    err, lerr = np.abs(o - o_ref), np.abs(lse - lse_ref)
    assert err.max() <= MAX_O and err.mean() <= MEAN_O and lerr.max() <= MAX_LSE, (err.max(), err.mean(), lerr.max())


@pytest.mark.gpu
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("B,H,N,d,causal,groups", [(1, 5, 200, 64, True, 3), (2, 3, 129, 128, False, 6),
                                                   (1, 1, 1, 64, False, 1), (3, 2, 384, 128, True, 0),
                                                   (1, 4, 1000, 64, True, 4)])
def test_host_forward_matches_oracle(B, H, N, d, causal, groups, pinned):
    q, k, v = make_inputs(B, H, N, d, seed=7000 + N + d + groups)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    scale = float(np.float32(1 / np.sqrt(d)))
    o, lse = fa.forward_host(q, k, v, scale=scale, causal=causal, n_groups=groups)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == 0
    assert not o.is_cuda and not lse.is_cuda
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    check(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("name,groups", [("b2_h32_n4096_d128_causal", 4), ("b4_h16_n2048_d128", 7),
                                         ("b16_h16_n1000_d64_causal_q8", 64), ("b1_h32_n16384_d128_causal", 0)])
def test_host_forward_bit_identical_to_device_forward(name, groups):
    w = WORKLOADS[name]
    q, k, v = (t.pin_memory() for t in workload_inputs(w))
    o_h, lse_h = fa.forward_host(q, k, v, scale=w.scale, causal=w.causal, n_groups=groups)
    o_d, lse_d = fa.forward(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    # and against the oracle on sampled rows
    rows = sample_rows(w.B, w.H, w.N, per_head=8, seed=w.seed)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal, rows=rows)
    check(o_h.double().numpy().reshape(-1, w.d)[rows], lse_h.double().numpy().reshape(-1)[rows], o_ref, lse_ref)


@pytest.mark.gpu
def test_back_to_back_calls_reuse_staging_in_order():
    B, H, N, d = 1, 8, 1024, 128
    scale = float(np.float32(1 / np.sqrt(d)))
    staging = fa.host_staging((B, H, N, d), torch.device("cuda"))
    ins = [tuple(t.pin_memory() for t in make_inputs(B, H, N, d, seed=s)) for s in (11, 12)]
    outs = [fa.forward_host(*x, scale=scale, causal=True, staging=staging, n_groups=4) for x in ins]
    torch.cuda.synchronize()
    for (q, k, v), (o, lse) in zip(ins, outs):
        o_ref, lse_ref = oracle.attention(q, k, v, scale, True)
        check(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref)


@pytest.mark.gpu
def test_device_pointer_refused_as_host_buffer():
    B, H, N, d = 1, 2, 128, 64
    dq = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    st = fa.host_staging((B, H, N, d), torch.device("cuda"))
    hq, hk, hv, ho = (torch.empty((B, H, N, d), dtype=torch.bfloat16) for _ in range(4))
    hl = torch.empty((B, H, N), dtype=torch.float32)
    good = [hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(), hl.data_ptr()] + [t.data_ptr() for t in st]
    # a device pointer where the host Q belongs
    args = list(good)
    args[0] = dq.data_ptr()
    assert fa.fa_fwd_host(*args, B, H, N, d, 0.125, False, 0, 0) == 1
    # a host pointer where the device staging Q belongs
    args = list(good)
    args[5] = hq.data_ptr()
    assert fa.fa_fwd_host(*args, B, H, N, d, 0.125, False, 0, 0) == 1
    # the same arguments with every pointer in its place are accepted
    assert fa.fa_fwd_host(*good, B, H, N, d, 0.125, False, 0, 0) == 0
    torch.cuda.synchronize()
