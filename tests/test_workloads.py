"""The seeded input generator: deterministic, the right shapes and values."""
import math

import numpy as np
import torch

from exact_attention_32_gb300.workloads import (HEADLINE, WORKLOADS, make_inputs,
                                                sample_rows, workload_inputs)


def test_deterministic_per_seed():
    a = make_inputs(2, 3, 17, 8, seed=5)
    b = make_inputs(2, 3, 17, 8, seed=5)
    c = make_inputs(2, 3, 17, 8, seed=6)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])


def test_shapes_and_dtype():
    q, k, v = make_inputs(2, 3, 17, 8, seed=5)
    for t in (q, k, v):
        assert t.shape == (2, 3, 17, 8) and t.dtype == torch.bfloat16 and t.is_contiguous()
    assert not torch.equal(q, k) and not torch.equal(k, v)


def test_q_gain_is_exact_power_of_two():
    q1, k1, v1 = make_inputs(1, 2, 64, 16, seed=9)
    q8, k8, v8 = make_inputs(1, 2, 64, 16, seed=9, q_gain=8.0)
    assert torch.equal(q8.float(), q1.float() * 8)
    assert torch.equal(k8, k1) and torch.equal(v8, v1)


def test_standard_normal_moments():
    q, k, v = make_inputs(1, 4, 4096, 64, seed=10)
    for t in (q, k, v):
        x = t.float()
        assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1) < 0.01


def test_workload_table():
    assert HEADLINE in WORKLOADS
    w = WORKLOADS[HEADLINE]
    assert (w.B, w.H, w.N, w.d, w.causal) == (1, 32, 16384, 128, True)
    assert w.flops == 4 * 32 * 16384 ** 2 * 128 / 2
    assert w.scale == float(np.float32(1 / math.sqrt(128)))
    stress = WORKLOADS["b16_h16_n1000_d64_causal_q8"]
    assert stress.q_gain == 8.0 and stress.N % 128 != 0
    q, k, v = workload_inputs(WORKLOADS["b1_h1_n256_d64"])
    assert q.shape == (1, 1, 256, 64)


def test_sample_rows_cover_boundaries():
    rows = sample_rows(2, 3, 1000, per_head=40, seed=1)
    assert np.all(np.diff(rows) > 0)
    for bh in range(6):
        sl = rows[(rows >= bh * 1000) & (rows < (bh + 1) * 1000)] - bh * 1000
        assert 0 in sl and 999 in sl and 127 in sl and 128 in sl
        assert len(sl) >= 40
