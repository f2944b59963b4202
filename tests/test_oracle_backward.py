"""Pins for the backward oracle (CPU): the gradient of sum(O * dO) checked
against what fixes it independently of the formulas the oracle restates.

  autograd          - fp64 torch autograd of the plain forward definition
  finite differences- central differences of an fp64 forward on tiny inputs
  identity          - rowsum(dP * P) = rowsum(dO * O) ("6.1 FlashAttention V1 in
                      detail", section 6.1)
  closed forms      - N = 1: dQ = dK = 0, dV = dO; causal row 0 of dQ is 0
  invariants        - adding one vector to every V row, or to every K row,
                      changes no gradient; rows of dS sum to zero
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_32_gb300.workloads import make_inputs


def inputs(B, H, N, d, seed, q_gain=1.0):
    q, k, v = make_inputs(B, H, N, d, seed=seed, q_gain=q_gain)
    g = torch.Generator().manual_seed(seed + 77)
    do = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)
    return q, k, v, do


def torch_reference(q, k, v, do, scale, causal):
    qd, kd, vd = (t.double().requires_grad_(True) for t in (q, k, v))
    s = scale * qd @ kd.transpose(-1, -2)
    if causal:
        N = q.shape[2]
        s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ vd
    (o * do.double()).sum().backward()
    return qd.grad.numpy(), kd.grad.numpy(), vd.grad.numpy(), o.detach().numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,scale", [(1, 4, 0.5), (7, 3, 0.7), (64, 16, 0.25), (130, 64, 0.125)])
def test_matches_autograd(N, d, scale, causal):
    q, k, v, do = inputs(2, 2, N, d, seed=N + d, q_gain=2.0)
    g = oracle.attention_backward(q, k, v, do, scale, causal)
    dq, dk, dv, o = torch_reference(q, k, v, do, scale, causal)
    shape = (4, N, d)
    for name, ref in (("dq", dq), ("dk", dk), ("dv", dv), ("o", o)):
        assert np.allclose(g[name], ref.reshape(shape), rtol=1e-10, atol=1e-12), name


@pytest.mark.parametrize("causal", [False, True])
def test_matches_central_differences(causal):
    N, d, scale = 5, 3, 0.6
    q, k, v, do = inputs(1, 1, N, d, seed=42, q_gain=1.5)
    g = oracle.attention_backward(q, k, v, do, scale, causal)
    X = {n: t.double().numpy()[0, 0] for n, t in (("q", q), ("k", k), ("v", v))}
    dO = do.double().numpy()[0, 0]

    def loss(Q, K, V):
        S = scale * Q @ K.T
        if causal:
            S = np.where(np.tril(np.ones((N, N), dtype=bool)), S, -np.inf)
        P = np.exp(S - S.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        return float(((P @ V) * dO).sum())

    h = 1e-6
    for name, grad in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        fd = np.zeros((N, d))
        for i in range(N):
            for c in range(d):
                args = dict(X)
                plus, minus = X[name].copy(), X[name].copy()
                plus[i, c] += h
                minus[i, c] -= h
                fd[i, c] = (loss(**{**{"Q": X["q"], "K": X["k"], "V": X["v"]},
                                    name.upper(): plus}) -
                            loss(**{**{"Q": X["q"], "K": X["k"], "V": X["v"]},
                                    name.upper(): minus})) / (2 * h)
        assert np.allclose(g[grad][0], fd, rtol=1e-6, atol=1e-8), name


@pytest.mark.parametrize("causal", [False, True])
def test_rowsum_identity(causal):
    q, k, v, do = inputs(1, 2, 40, 8, seed=3)
    g = oracle.attention_backward(q, k, v, do, 0.3, causal)
    # D = rowsum(dO * O) must equal rowsum(dP * P); rebuild P and dP independently
    for bh in range(2):
        Q, K, V, dO = (t.double().numpy().reshape(2, 40, 8)[bh] for t in (q, k, v, do))
        S = 0.3 * Q @ K.T
        if causal:
            S = np.where(np.tril(np.ones((40, 40), dtype=bool)), S, -np.inf)
        P = np.exp(S - g["lse"][bh][:, None])
        dP = dO @ V.T
        assert np.allclose((dP * P).sum(1), g["D"][bh], rtol=1e-12, atol=1e-12)
        assert np.allclose(P.sum(1), 1.0, rtol=0, atol=1e-12)


def test_single_key_closed_form():
    q, k, v, do = inputs(2, 2, 1, 16, seed=5)
    g = oracle.attention_backward(q, k, v, do, 0.5, False)
    assert np.all(g["dq"] == 0) and np.all(g["dk"] == 0)
    assert np.array_equal(g["dv"], do.double().numpy().reshape(4, 1, 16))


def test_causal_first_row_has_no_query_gradient():
    # row 0 sees only key 0: P = 1, dS = 0
    q, k, v, do = inputs(1, 1, 20, 8, seed=6)
    g = oracle.attention_backward(q, k, v, do, 0.5, True)
    assert np.allclose(g["dq"][0, 0], 0.0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("which", ["v", "k"])
def test_shift_invariance(which, causal):
    # the same vector added to every V row (or every K row) leaves all three gradients unchanged
    q, k, v, do = inputs(1, 2, 30, 8, seed=9)
    shift = torch.tensor([1.0, -2.0, 0.5, 4.0, -1.0, 0.25, 2.0, -0.5]).to(torch.bfloat16)
    base = oracle.attention_backward(q, k, v, do, 0.4, causal)
    # small exactly representable values so the shifted inputs are exact in bf16
    if which == "v":
        v2 = (v.float().round() + shift.float()).to(torch.bfloat16)
        v1 = v.float().round().to(torch.bfloat16)
        a = oracle.attention_backward(q, k, v1, do, 0.4, causal)
        b = oracle.attention_backward(q, k, v2, do, 0.4, causal)
    else:
        k2 = (k.float().round() + shift.float()).to(torch.bfloat16)
        k1 = k.float().round().to(torch.bfloat16)
        a = oracle.attention_backward(q, k1, v, do, 0.4, causal)
        b = oracle.attention_backward(q, k2, v, do, 0.4, causal)
    for name in ("dq", "dk", "dv"):
        assert np.allclose(a[name], b[name], rtol=1e-9, atol=1e-10), name
    assert base["dq"].shape == (2, 30, 8)


def test_rows_of_ds_sum_to_zero():
    q, k, v, do = inputs(1, 1, 50, 8, seed=10)
    g = oracle.attention_backward(q, k, v, do, 0.5, True)
    # dQ_i = scale * sum_j dS_ij k_j; with every k_j = 1 (all ones) dQ must vanish
    ones = torch.ones_like(k)
    g1 = oracle.attention_backward(q, ones, v, do, 0.5, True)
    assert np.allclose(g1["dq"], 0.0, atol=1e-12)
    assert g["dq"].shape == (1, 50, 8)


def test_slice_selection():
    q, k, v, do = inputs(2, 3, 33, 8, seed=11)
    full = oracle.attention_backward(q, k, v, do, 0.5, True)
    part = oracle.attention_backward(q, k, v, do, 0.5, True, slices=[4, 1])
    for name in ("dq", "dk", "dv", "lse"):
        assert np.array_equal(part[name], full[name][[4, 1]])
