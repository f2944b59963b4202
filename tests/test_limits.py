"""Sizes and inputs at the edges of what the forward handles.

GPU: a 131072-token sequence (causal and not, both head sizes; sampled rows
against the fp64 oracle, every value finite); 4096 (b, h) slices of 64 rows
each (every row against the oracle); split-KV at the long length; and Q = 0,
where every admitted key has the same weight, so O is the mean of the
admitted V rows (causal: the prefix mean) and LSE = ln(number of admitted
keys), a closed form checked without the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_32_gb300 as fa
from exact_attention_32_gb300 import make_inputs
from exact_attention_32_gb300.workloads import sample_rows

MAX_O, MEAN_O, MAX_LSE = 2e-2, 2e-3, 1e-3


def check(o, lse, o_ref, lse_ref):
    err, lerr = np.abs(o - o_ref), np.abs(lse - lse_ref)
    assert err.max() <= MAX_O and err.mean() <= MEAN_O and lerr.max() <= MAX_LSE, (err.max(), err.mean(), lerr.max())


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_sampled_rows(causal, d):
    B, H, N = 1, 1, 131072
    q, k, v = make_inputs(B, H, N, d, seed=9000 + d + causal)
    scale = float(np.float32(1 / np.sqrt(d)))
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == 0
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = sample_rows(B, H, N, per_head=24, seed=9)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal, rows=rows)
    check(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_many_short_slices_every_row(causal):
    B, H, N, d = 64, 64, 64, 64
    q, k, v = make_inputs(B, H, N, d, seed=9100 + causal)
    scale = float(np.float32(1 / np.sqrt(d)))
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == 0
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref)


@pytest.mark.gpu
def test_splitkv_long_sequence_sampled_rows():
    B, H, N, d = 1, 1, 131072, 128
    q, k, v = make_inputs(B, H, N, d, seed=9200)
    scale = float(np.float32(1 / np.sqrt(d)))
    o, lse, _ = fa.forward_splitkv(q.cuda(), k.cuda(), v.cuda(), 8, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == 0
    rows = sample_rows(B, H, N, per_head=16, seed=10)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, True, rows=rows)
    check(o.double().cpu().numpy().reshape(-1, d)[rows], lse.double().cpu().numpy().reshape(-1)[rows], o_ref, lse_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_the_mean_of_admitted_values(causal, d):
    # q = 0: every logit is 0, so each admitted key has weight 1 / (number admitted)
    B, H, N = 2, 3, 700
    _, k, v = make_inputs(B, H, N, d, seed=9300 + d)
    q = torch.zeros_like(k)
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    vd = v.double().numpy()
    if causal:
        counts = np.arange(1, N + 1, dtype=np.float64)
        o_ref = np.cumsum(vd, axis=2) / counts[:, None]
    else:
        counts = np.full(N, float(N))
        o_ref = np.broadcast_to(vd.mean(axis=2, keepdims=True), vd.shape)
    lse_ref = np.broadcast_to(np.log(counts), (B, H, N))
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref)
