"""Block-sparse forward (fa_fwd_blocksparse) against the fp64 oracle: every
row, forward tolerances (max |dO| <= 2e-2, mean |dO| <= 2e-3, max |dLSE| <= 1e-3)
on rows that admit keys; rows that admit none must be exactly O = 0, LSE = -inf."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_32_gb300 import fa_get_device_status, forward_blocksparse, make_inputs

pytestmark = pytest.mark.gpu


def run_and_check(q, k, v, scale, causal, mask):
    o, lse = forward_blocksparse(q.cuda(), k.cuda(), v.cuda(), torch.as_tensor(mask), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa_get_device_status(0) == 0
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    o_ref, lse_ref = oracle.attention_blocksparse(q, k, v, scale, causal, mask)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(o[empty] == 0.0)
    if (~empty).any():
        e, le = np.abs(o[~empty] - o_ref[~empty]), np.abs(lse[~empty] - lse_ref[~empty])
        assert e.max() <= 2e-2 and e.mean() <= 2e-3 and le.max() <= 1e-3, (e.max(), e.mean(), le.max())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,density", [(128, 1.0), (300, 0.5), (1000, 0.3), (1000, 0.7), (640, 0.0)])
def test_random_masks(N, density, d, causal):
    nb = -(-N // 128)
    rng = np.random.default_rng(N + int(10 * density) + d)
    mask = (rng.random((nb, nb)) < density).astype(np.uint8)
    q, k, v = make_inputs(2, 2, N, d, seed=5000 + N + d + causal)
    run_and_check(q, k, v, float(np.float32(1 / np.sqrt(d))), causal, mask)


@pytest.mark.parametrize("causal", [False, True])
def test_local_window_plus_global_columns(causal):
    # a sliding window of 3 blocks plus the first block as global keys, N = 4096
    nb = 32
    i, j = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    mask = ((np.abs(i - j) <= 1) | (j == 0)).astype(np.uint8)
    q, k, v = make_inputs(1, 2, 4096, 128, seed=5100 + causal)
    run_and_check(q, k, v, 0.0883883461356163, causal, mask)


def test_diagonal_blocks_and_empty_rows():
    mask = np.eye(4, dtype=np.uint8)
    mask[2, 2] = 0  # query block 2 admits nothing
    q, k, v = make_inputs(1, 3, 500, 64, seed=5200)
    run_and_check(q, k, v, 0.125, False, mask)
