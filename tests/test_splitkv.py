"""Split-KV forward and the merge of partial (O, LSE) results.

CPU: the workspace-size rule and argument rejection (no device call).
GPU: fa_fwd_splitkv against the dense fp64 oracle; every per-range part it
leaves in the workspace against the oracle restricted to that key range; and
fa_combine against the oracle's two-block merge on seeded synthetic parts.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_32_gb300 import build as fa_build
from exact_attention_32_gb300 import (WORKLOADS, combine, fa_get_device_status, forward_splitkv,
                                      make_inputs, workload_inputs)
from exact_attention_32_gb300.workloads import sample_rows

MAX_O, MEAN_O, MAX_LSE = 2e-2, 2e-3, 1e-3


def geometry(N, n_splits):
    per = -(-N // n_splits)
    chunk = -(-per // 128) * 128
    return chunk, -(-N // chunk)


@pytest.fixture(scope="module")
def libfa():
    L = ctypes.CDLL(fa_build.build())
    i64 = ctypes.c_int64
    L.fa_fwd_splitkv_workspace_bytes.restype = i64
    L.fa_fwd_splitkv_workspace_bytes.argtypes = [i64] * 5
    vp = ctypes.c_void_p
    L.fa_fwd_splitkv.restype = ctypes.c_int
    L.fa_fwd_splitkv.argtypes = [vp] * 5 + [i64] * 4 + [ctypes.c_float, ctypes.c_int, i64, vp, i64, vp]
    return L


@pytest.mark.parametrize("B,H,N,d,S", [(1, 1, 1000, 64, 3), (2, 3, 256, 128, 2), (1, 2, 16384, 128, 4),
                                       (1, 1, 100, 64, 32), (3, 1, 129, 128, 1)])
def test_workspace_bytes(libfa, B, H, N, d, S):
    chunk, parts = geometry(N, S)
    assert chunk % 128 == 0 and (parts - 1) * chunk < N <= parts * chunk and parts <= S
    assert libfa.fa_fwd_splitkv_workspace_bytes(B, H, N, d, S) == parts * B * H * N * (d + 1) * 4


@pytest.mark.parametrize("args", [(1, 1, 256, 64, 0), (1, 1, 256, 64, 33), (1, 1, 0, 64, 2), (1, 1, 256, 96, 2)])
def test_workspace_bytes_rejects(libfa, args):
    assert libfa.fa_fwd_splitkv_workspace_bytes(*args) == -1


def test_small_workspace_rejected_before_any_device_call(libfa):
    need = libfa.fa_fwd_splitkv_workspace_bytes(1, 1, 256, 64, 2)
    assert libfa.fa_fwd_splitkv(16, 16, 16, 16, 16, 1, 1, 256, 64, 0.125, 0, 2, 16, need - 16, None) == 1
    assert libfa.fa_fwd_splitkv(16, 16, 16, 16, 16, 1, 1, 256, 64, 0.125, 0, 40, 16, need, None) == 1


def check(o, lse, o_ref, lse_ref):
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err, lerr = np.abs(o - o_ref), np.abs(lse - lse_ref)
    assert err.max() <= MAX_O and err.mean() <= MEAN_O and lerr.max() <= MAX_LSE, \
        (err.max(), err.mean(), lerr.max())


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,S", [(1, 2), (200, 2), (300, 3), (1000, 3), (1000, 8), (640, 5)])
def test_splitkv_matches_dense_and_parts_match_ranges(N, S, d, causal):
    q, k, v = make_inputs(2, 2, N, d, seed=500 + N + S + d + causal)
    scale = float(np.float32(1 / np.sqrt(d)))
    o, lse, ws = forward_splitkv(q.cuda(), k.cuda(), v.cuda(), S, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa_get_device_status(0) == 0
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref)
    # the parts in the workspace: each is the attention over its key range alone
    chunk, parts = geometry(N, S)
    rows = 2 * 2 * N
    wsf = ws.view(torch.float32).cpu().double().numpy()
    o_parts = wsf[: parts * rows * d].reshape(parts, 2, 2, N, d)
    lse_parts = wsf[parts * rows * d: parts * rows * (d + 1)].reshape(parts, 2, 2, N)
    for s in range(parts):
        lo, hi = s * chunk, min((s + 1) * chunk, N)
        op_ref, lp_ref = oracle.attention(q, k, v, scale, causal, kv_range=(lo, hi))
        empty = np.isneginf(lp_ref)
        assert np.array_equal(np.isneginf(lse_parts[s]), empty)
        assert np.all(o_parts[s][empty] == 0.0)
        if (~empty).any():
            err = np.abs(o_parts[s][~empty] - op_ref[~empty])
            assert err.max() <= MAX_O and err.mean() <= MEAN_O
            assert np.abs(lse_parts[s][~empty] - lp_ref[~empty]).max() <= MAX_LSE


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 5, 32])
def test_combine_matches_oracle_merge(S, d):
    # seeded synthetic parts, including parts with no admitted key (LSE = -inf, O = 0)
    g = torch.Generator().manual_seed(S * 1000 + d)
    B, H, N = 2, 3, 77
    o_parts = torch.randn((S, B, H, N, d), generator=g, dtype=torch.float32)
    lse_parts = torch.randn((S, B, H, N), generator=g, dtype=torch.float32) * 20
    drop = torch.rand((S, B, H, N), generator=g) < 0.3
    drop[0, 0, 0, :5] = True
    if S > 1:
        drop[1:, 0, 0, :3] = True  # rows 0-2 of (0, 0): no key in any part
    lse_parts[drop] = float("-inf")
    o_parts[drop.unsqueeze(-1).expand_as(o_parts)] = 0.0
    o, lse = combine(o_parts.cuda(), lse_parts.cuda())
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.merge(o_parts.double().numpy(), lse_parts.double().numpy())
    og, lg = o.double().cpu().numpy(), lse.double().cpu().numpy()
    none = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), none)
    assert np.all(og[none] == 0.0)
    assert np.abs(og - o_ref).max() <= 2 ** -8 * max(1.0, np.abs(o_ref).max())
    assert np.abs(lg[~none] - lse_ref[~none]).max() <= 1e-4


@pytest.mark.gpu
@pytest.mark.parametrize("name,S", [("b4_h16_n2048_d128", 4), ("b1_h32_n16384_d128_causal", 4),
                                    ("b1_h1_n256_d64", 2)])
def test_splitkv_workloads_sampled_rows(name, S):
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)
    o, lse, _ = forward_splitkv(q.cuda(), k.cuda(), v.cuda(), S, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.H, w.N, per_head=16, seed=w.seed)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal, rows=rows)
    check(o.double().cpu().numpy().reshape(-1, w.d)[rows], lse.double().cpu().numpy().reshape(-1)[rows],
          o_ref, lse_ref)
