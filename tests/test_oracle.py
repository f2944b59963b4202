"""Pins for the oracle: what the pages and the mathematics fix, not the oracle
restated.  CPU only.

Each pin targets a class of mistake:
  worked example            - the merge algebra and the value the page prints
  decimal brute force       - any wrong index, transposed operand, sign, scale
                              or causal direction (different formulation: no
                              max shift, 50 digits)
  closed forms              - N = 1, causal row 0, equal keys, q = 0
  rows of P sum to one      - the normalisation (pass 3)
  invariants                - permutation, linearity in V, logit shift vs LSE
  online vs dense           - tile size / order invariance of the (m, l, u) merge
  negative test             - the K/V out-of-range mask matters
  large logits              - max subtraction keeps the result finite and exact
  key ranges and merge      - partials over disjoint key ranges, folded with the
                              two-block merge, give dense attention (the worked
                              example in both orders; random splits)
"""
import math
import os
from decimal import Decimal

import numpy as np
import pytest
import torch

import oracle
from exact_attention_32_gb300.workloads import WORKLOADS, make_inputs, workload_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [float(x) for x in vals]
    return out


def worked_example_inputs():
    g = read_golden("worked_example.txt")
    n = len(g["scores"])
    # every query row is q = [1] against keys = the printed scores, scale 1
    q = bf16(np.ones((1, 1, n, 1)))
    k = bf16(np.asarray(g["scores"]).reshape(1, 1, n, 1))
    v = bf16(np.asarray(g["values"]).reshape(1, 1, n, 1))
    return g, q, k, v


# --------------------------------------------------------------- worked example

def test_worked_example_dense():
    g, q, k, v = worked_example_inputs()
    o, lse = oracle.attention(q, k, v, 1.0, False)
    tol = 0.5 * 10 ** -int(g["digits"][0])
    assert np.all(np.abs(o[..., 0] - g["output"][0]) <= tol)
    # LSE closed form for scores [2, 1, 0]: 2 + ln(1 + e^-1 + e^-2)
    assert np.allclose(lse, 2.0 + math.log(1 + math.exp(-1) + math.exp(-2)), rtol=0, atol=1e-14)


@pytest.mark.parametrize("order", [[0, 1], [1, 0]])
def test_worked_example_online_both_orders(order):
    g, q, k, v = worked_example_inputs()
    # tiles [2, 1] | [0]: block_k = 2, visited in both orders
    o, lse = oracle.attention_online(q, k, v, 1.0, False, block_q=3, block_k=2, order=order)
    tol = 0.5 * 10 ** -int(g["digits"][0])
    assert np.all(np.abs(o[..., 0] - g["output"][0]) <= tol)
    o_d, lse_d = oracle.attention(q, k, v, 1.0, False)
    assert np.allclose(o, o_d, rtol=0, atol=1e-15)
    assert np.allclose(lse, lse_d, rtol=0, atol=1e-15)


def test_worked_example_first_tile_state():
    # after tile [2, 1] alone: m = 2, l = 1 + e^-1, u = 1 + 3 e^-1
    q = bf16(np.ones((1, 1, 2, 1)))
    k = bf16(np.asarray([2.0, 1.0]).reshape(1, 1, 2, 1))
    v = bf16(np.asarray([1.0, 3.0]).reshape(1, 1, 2, 1))
    o, lse = oracle.attention(q, k, v, 1.0, False)
    e1 = math.exp(-1)
    assert np.allclose(o[..., 0], (1 + 3 * e1) / (1 + e1), rtol=0, atol=1e-15)
    assert np.allclose(lse, 2 + math.log(1 + e1), rtol=0, atol=1e-15)


def test_worked_example_decimal():
    g, q, k, v = worked_example_inputs()
    O, L = oracle.attention_decimal(q, k, v, 1, False)
    assert abs(float(O[0][0][0][0]) - g["output"][0]) <= 0.5e-6
    e = [Decimal(x).exp() for x in (2, 1, 0)]
    assert abs(O[0][0][0][0] - (e[0] * 1 + e[1] * 3 + e[2] * 5) / sum(e)) < Decimal("1e-45")


# ---------------------------------------------------------- decimal brute force

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,scale", [(1, 1, 1.0), (3, 2, 0.5), (5, 4, 0.7071067690849304),
                                       (8, 3, 1.25)])
def test_dense_matches_decimal_brute_force(causal, N, d, scale):
    q, k, v = make_inputs(2, 2, N, d, seed=7 + N * 10 + d)
    o, lse = oracle.attention(q, k, v, scale, causal)
    O, L = oracle.attention_decimal(q, k, v, scale, causal)
    Od = np.array([[[[float(x) for x in r] for r in hh] for hh in bb] for bb in O])
    Ld = np.array([[[float(x) for x in hh] for hh in bb] for bb in L])
    assert np.allclose(o, Od, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, Ld, rtol=1e-12, atol=1e-13)


def test_decimal_catches_transposed_scores():
    # a plausible mistake - S_ji instead of S_ij - must not agree with brute force
    q, k, v = make_inputs(1, 1, 5, 3, seed=3)
    o, _ = oracle.attention(k, q, v, 1.0, True)  # swapped roles
    O, _ = oracle.attention_decimal(q, k, v, 1.0, True)
    Od = np.array([[[[float(x) for x in r] for r in hh] for hh in bb] for bb in O])
    assert not np.allclose(o, Od, rtol=1e-6, atol=1e-6)


# ----------------------------------------------------------------- closed forms

@pytest.mark.parametrize("d", [1, 64, 128])
def test_single_key_returns_its_value(d):
    # N = 1: O = v_0 exactly, LSE = s_00
    q, k, v = make_inputs(2, 3, 1, d, seed=11)
    scale = 0.3
    o, lse = oracle.attention(q, k, v, scale, False)
    assert np.array_equal(o, v.to(torch.float64).numpy())
    s = scale * np.einsum("bhnc,bhnc->bhn", q.to(torch.float64).numpy(), k.to(torch.float64).numpy())
    assert np.allclose(lse, s, rtol=1e-14, atol=1e-14)


def test_causal_row0_is_v0():
    q, k, v = make_inputs(2, 2, 9, 16, seed=12)
    o, lse = oracle.attention(q, k, v, 0.25, True)
    assert np.array_equal(o[:, :, 0, :], v[:, :, 0, :].to(torch.float64).numpy())
    s00 = 0.25 * np.einsum("bhc,bhc->bh", q[:, :, 0].to(torch.float64).numpy(),
                           k[:, :, 0].to(torch.float64).numpy())
    assert np.allclose(lse[:, :, 0], s00, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_keys_give_mean_of_values(causal):
    # all K rows equal -> every admitted key has the same logit s:
    # O_i = mean of V over admitted keys, LSE_i = s + ln|A(i)|
    B, H, N, d = 1, 2, 37, 8
    q, _, v = make_inputs(B, H, N, d, seed=13)
    krow = make_inputs(1, 1, 1, d, seed=14)[0]
    k = krow.expand(B, H, N, d).contiguous()
    scale = 0.5
    o, lse = oracle.attention(q, k, v, scale, causal)
    vd = v.to(torch.float64).numpy()
    s = scale * np.einsum("bhnc,c->bhn", q.to(torch.float64).numpy(),
                          krow.to(torch.float64).numpy().reshape(-1))
    for i in range(N):
        n = i + 1 if causal else N
        assert np.allclose(o[:, :, i], vd[:, :, :n].mean(axis=2), rtol=1e-12, atol=1e-13)
        assert np.allclose(lse[:, :, i], s[:, :, i] + math.log(n), rtol=1e-13, atol=1e-13)


def test_zero_query_is_uniform():
    B, H, N, d = 1, 1, 50, 4
    _, k, v = make_inputs(B, H, N, d, seed=15)
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
    o, lse = oracle.attention(q, k, v, 1.0, False)
    assert np.allclose(o, v.to(torch.float64).numpy().mean(axis=2, keepdims=True).repeat(N, 2),
                       rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, math.log(N), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    # a V column of ones comes out as ones: sum_j P_ij = 1
    q, k, v = make_inputs(2, 2, 64, 8, seed=16, q_gain=4.0)
    v = v.clone()
    v[..., 3] = 1.0
    o, _ = oracle.attention(q, k, v, 0.35, causal)
    assert np.allclose(o[..., 3], 1.0, rtol=0, atol=1e-13)


# ------------------------------------------------------------------- invariants

def test_permuting_keys_and_values_together():
    q, k, v = make_inputs(1, 2, 40, 8, seed=17)
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(1))
    o1, l1 = oracle.attention(q, k, v, 0.4, False)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-13)
    assert np.allclose(l1, l2, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_linear_in_values(causal):
    # small-integer V so that V1 + V2 is exact in bf16
    q, k, _ = make_inputs(1, 2, 33, 8, seed=18)
    rng = np.random.default_rng(0)
    v1 = bf16(rng.integers(-8, 9, size=(1, 2, 33, 8)))
    v2 = bf16(rng.integers(-8, 9, size=(1, 2, 33, 8)))
    o1, _ = oracle.attention(q, k, v1, 0.5, causal)
    o2, _ = oracle.attention(q, k, v2, 0.5, causal)
    o12, _ = oracle.attention(q, k, bf16((v1.float() + v2.float()).numpy()), 0.5, causal)
    assert np.allclose(o12, o1 + o2, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_logit_shift_moves_only_lse(causal):
    # an extra feature column: q gets t = 4, k gets 1 -> every logit of the row
    # grows by scale * 4 = 2; O is unchanged, LSE grows by exactly 2
    B, H, N, d = 1, 2, 30, 6
    q, k, v = make_inputs(B, H, N, d, seed=19)
    q2 = torch.cat([q, torch.full((B, H, N, 1), 4.0, dtype=torch.bfloat16)], dim=-1)
    k2 = torch.cat([k, torch.ones((B, H, N, 1), dtype=torch.bfloat16)], dim=-1)
    v2 = torch.cat([v, torch.zeros((B, H, N, 1), dtype=torch.bfloat16)], dim=-1)
    o1, l1 = oracle.attention(q, k, v, 0.5, causal)
    o2, l2 = oracle.attention(q2, k2, v2, 0.5, causal)
    assert np.allclose(o2[..., :d], o1, rtol=1e-12, atol=1e-13)
    assert np.allclose(l2, l1 + 2.0, rtol=0, atol=1e-12)


def test_row_subset_is_identical_to_full():
    q, k, v = make_inputs(2, 3, 50, 16, seed=20)
    o, lse = oracle.attention(q, k, v, 0.25, True)
    rows = np.array([0, 49, 50, 123, 299], dtype=np.int64)
    os_, ls = oracle.attention(q, k, v, 0.25, True, rows=rows)
    assert np.array_equal(os_, o.reshape(-1, 16)[rows])
    assert np.array_equal(ls, lse.reshape(-1)[rows])


# ------------------------------------------------------------- online vs dense

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block_q,block_k", [(7, 1), (16, 3), (5, 7), (64, 64), (32, 128), (100, 100)])
def test_online_equals_dense_any_tile_size(causal, block_q, block_k):
    q, k, v = make_inputs(1, 2, 100, 16, seed=21, q_gain=3.0)
    od, ld = oracle.attention(q, k, v, 0.25, causal)
    oo, lo = oracle.attention_online(q, k, v, 0.25, causal, block_q, block_k)
    assert np.allclose(oo, od, rtol=1e-12, atol=1e-12)
    assert np.allclose(lo, ld, rtol=1e-13, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("how", ["reversed", "random"])
def test_online_equals_dense_any_tile_order(causal, how):
    N, bk = 77, 8
    q, k, v = make_inputs(2, 1, N, 8, seed=22, q_gain=4.0)
    t_c = -(-N // bk)
    order = list(range(t_c))[::-1] if how == "reversed" else \
        list(np.random.default_rng(5).permutation(t_c))
    od, ld = oracle.attention(q, k, v, 0.5, causal)
    oo, lo = oracle.attention_online(q, k, v, 0.5, causal, 16, bk, order=order)
    assert np.allclose(oo, od, rtol=1e-12, atol=1e-12)
    assert np.allclose(lo, ld, rtol=1e-13, atol=1e-12)


def test_tiny_workload_tile_order_invariance():
    # the 1x1x256x64 workload: online merge in a random K/V-tile order matches dense
    w = WORKLOADS["b1_h1_n256_d64"]
    q, k, v = workload_inputs(w)
    od, ld = oracle.attention(q, k, v, w.scale, w.causal)
    order = list(np.random.default_rng(9).permutation(256 // 32))
    oo, lo = oracle.attention_online(q, k, v, w.scale, w.causal, 64, 32, order=order)
    assert np.allclose(oo, od, rtol=1e-12, atol=1e-12)
    assert np.allclose(lo, ld, rtol=1e-13, atol=1e-12)


def test_missing_tail_mask_is_caught():
    # ragged N with zero-padded K/V rows let into the softmax must NOT match
    N = 1000
    q, k, v = make_inputs(1, 2, N, 16, seed=23)
    od, ld = oracle.attention(q, k, v, 0.25, False)
    ob, lb = oracle.attention_online(q, k, v, 0.25, False, 128, 128, mask_tail=False)
    assert np.max(np.abs(lb - ld)) > 1e-3
    assert np.max(np.abs(ob - od)) > 1e-4
    og, lg = oracle.attention_online(q, k, v, 0.25, False, 128, 128, mask_tail=True)
    assert np.allclose(og, od, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- large logits

def test_large_logits_match_unshifted_fp64():
    # Q scaled by 8 (logits up to about +-50): the oracle stays finite and agrees
    # with the unshifted softmax, which fp64 can still evaluate at this range
    q, k, v = make_inputs(1, 2, 300, 64, seed=24, q_gain=8.0)
    scale = float(np.float32(1 / 8))
    o, lse = oracle.attention(q, k, v, scale, True)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    qd, kd, vd = (t.to(torch.float64).numpy() for t in (q, k, v))
    s = scale * np.einsum("bhic,bhjc->bhij", qd, kd)
    assert np.abs(s).max() > 25
    mask = np.tril(np.ones((300, 300), dtype=bool))
    e = np.where(mask, np.exp(np.where(mask, s, 0.0)), 0.0)
    z = e.sum(-1)
    assert np.allclose(o, np.einsum("bhij,bhjc->bhic", e, vd) / z[..., None], rtol=1e-10, atol=1e-12)
    assert np.allclose(lse, np.log(z), rtol=1e-13, atol=1e-12)


def test_widening_is_exact():
    # bf16 extremes and subnormals go through the C oracle unchanged (N = 1: O = v)
    bits = np.array([0x0001, 0x8001, 0x007F, 0x0080, 0x3F80, 0xBF80, 0x7F7F, 0xFF7F,
                     0x4049, 0x3C23, 0x0000, 0x8000, 0x4000, 0xC2C8, 0x1234, 0x5678],
                    dtype=np.uint16)
    v = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(1, 1, 1, 16)
    q = torch.zeros((1, 1, 1, 16), dtype=torch.bfloat16)
    o, lse = oracle.attention(q, q, v, 1.0, False)
    assert np.array_equal(o.reshape(-1), v.to(torch.float64).numpy().reshape(-1))
    assert lse.reshape(-1)[0] == 0.0


def test_invalid_arguments_rejected():
    q, k, v = make_inputs(1, 1, 4, 2, seed=1)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, 1.0, False, rows=[4])
    with pytest.raises(ValueError):
        oracle.attention(q, k[:, :, :3], v, 1.0, False)


# ---------------------------------------------------- key ranges and the merge

@pytest.mark.parametrize("order", [[0, 1], [1, 0]])
def test_worked_example_by_partials_and_merge(order):
    # the page's split [2, 1] | [0] as two key ranges, merged in both orders
    g, q, k, v = worked_example_inputs()
    parts = [oracle.attention(q, k, v, 1.0, False, kv_range=r) for r in [(0, 2), (2, 3)]]
    parts = [parts[i] for i in order]
    o, lse = oracle.merge([p[0] for p in parts], [p[1] for p in parts])
    tol = 0.5 * 10 ** -int(g["digits"][0])
    assert np.all(np.abs(o[..., 0] - g["output"][0]) <= tol)
    assert np.allclose(lse, 2.0 + math.log(1 + math.exp(-1) + math.exp(-2)), rtol=0, atol=1e-14)
    # first part alone: m = 2, l = 1 + e^-1, u = 1 + 3 e^-1
    o1, l1 = parts[order.index(0)]
    assert np.allclose(o1[..., 0], (1 + 3 * math.exp(-1)) / (1 + math.exp(-1)), rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cuts", [[0, 50], [0, 17, 50], [0, 1, 2, 49, 50], [0, 25, 30, 31, 50]])
def test_merge_of_key_range_partials_is_dense(causal, cuts):
    q, k, v = make_inputs(2, 2, 50, 8, seed=31, q_gain=3.0)
    od, ld = oracle.attention(q, k, v, 0.4, causal)
    parts = [oracle.attention(q, k, v, 0.4, causal, kv_range=(a, b)) for a, b in zip(cuts[:-1], cuts[1:])]
    for perm in (list(range(len(parts))), list(range(len(parts)))[::-1]):
        o, lse = oracle.merge([parts[i][0] for i in perm], [parts[i][1] for i in perm])
        assert np.allclose(o, od, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse, ld, rtol=1e-13, atol=1e-12)


def test_single_key_range_returns_that_value():
    q, k, v = make_inputs(1, 2, 20, 8, seed=32)
    o, lse = oracle.attention(q, k, v, 0.5, False, kv_range=(7, 8))
    assert np.array_equal(o, np.broadcast_to(v[:, :, 7:8].to(torch.float64).numpy(), o.shape))
    s = 0.5 * np.einsum("bhic,bhc->bhi", q.to(torch.float64).numpy(), k[:, :, 7].to(torch.float64).numpy())
    assert np.allclose(lse, s, rtol=1e-14, atol=1e-14)


def test_rows_without_admitted_keys():
    # causal rows before the range start admit no key: O = 0, LSE = -inf,
    # and such a part carries no weight in the merge
    q, k, v = make_inputs(1, 1, 30, 4, seed=33)
    o, lse = oracle.attention(q, k, v, 0.5, True, kv_range=(10, 30))
    assert np.all(o[:, :, :10] == 0) and np.all(np.isneginf(lse[:, :, :10]))
    assert np.all(np.isfinite(lse[:, :, 10:]))
    o0, l0 = oracle.attention(q, k, v, 0.5, True, kv_range=(0, 10))
    om, lm = oracle.merge([o0, o], [l0, lse])
    od, ld = oracle.attention(q, k, v, 0.5, True)
    assert np.allclose(om, od, rtol=1e-12, atol=1e-12) and np.allclose(lm, ld, rtol=1e-13, atol=1e-12)


def test_merge_of_one_part_is_identity():
    rng = np.random.default_rng(3)
    o = rng.normal(size=(2, 3, 5, 4))
    lse = rng.normal(size=(2, 3, 5)) * 10
    om, lm = oracle.merge([o], [lse])
    assert np.allclose(om, o, rtol=0, atol=1e-15) and np.allclose(lm, lse, rtol=0, atol=1e-14)


def test_invalid_key_range_rejected():
    q, k, v = make_inputs(1, 1, 4, 2, seed=1)
    for r in [(2, 2), (-1, 3), (0, 5), (3, 1)]:
        with pytest.raises(ValueError):
            oracle.attention(q, k, v, 1.0, False, kv_range=r)


# ------------------------------------------------------------------ block-sparse

@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_all_ones_is_dense(causal):
    q, k, v = make_inputs(1, 2, 300, 16, seed=41)
    o, lse = oracle.attention_blocksparse(q, k, v, 0.25, causal, np.ones((3, 3)))
    od, ld = oracle.attention(q, k, v, 0.25, causal)
    assert np.allclose(o, od, rtol=1e-12, atol=1e-12) and np.allclose(lse, ld, rtol=1e-13, atol=1e-12)


def test_blocksparse_block_diagonal_is_per_block_attention():
    # a block-diagonal mask = independent attention inside each 128-row block
    N, d = 384, 16
    q, k, v = make_inputs(1, 2, N, d, seed=42)
    o, lse = oracle.attention_blocksparse(q, k, v, 0.25, False, np.eye(3))
    for b0 in range(0, N, 128):
        sl = slice(b0, b0 + 128)
        ob, lb = oracle.attention(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(), v[:, :, sl].contiguous(),
                                  0.25, False)
        assert np.allclose(o[:, :, sl], ob, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[:, :, sl], lb, rtol=1e-13, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_complementary_masks_merge_to_dense(causal):
    # two masks that split the admitted blocks between them merge back to dense
    rng = np.random.default_rng(7)
    N = 500
    nb = 4
    m1 = rng.random((nb, nb)) < 0.5
    q, k, v = make_inputs(1, 2, N, 8, seed=43, q_gain=2.0)
    a = oracle.attention_blocksparse(q, k, v, 0.5, causal, m1)
    b = oracle.attention_blocksparse(q, k, v, 0.5, causal, ~m1)
    o, lse = oracle.merge([a[0], b[0]], [a[1], b[1]])
    od, ld = oracle.attention(q, k, v, 0.5, causal)
    assert np.allclose(o, od, rtol=1e-12, atol=1e-12) and np.allclose(lse, ld, rtol=1e-13, atol=1e-12)


def test_blocksparse_row_without_blocks():
    q, k, v = make_inputs(1, 1, 256, 8, seed=44)
    mask = np.array([[1, 1], [0, 0]])
    o, lse = oracle.attention_blocksparse(q, k, v, 0.5, False, mask)
    assert np.all(o[:, :, 128:] == 0) and np.all(np.isneginf(lse[:, :, 128:]))
    assert np.all(np.isfinite(lse[:, :, :128]))


@pytest.mark.parametrize("name,head", [("b1_h1_n256_d64", (0, 0)), ("b16_h16_n1000_d64_causal_q8", (3, 7))])
def test_dense_matches_library_softmax_at_workload_size(name, head):
    # the textbook form with library routines: scores by a matrix product, a
    # library softmax along the keys, then another matrix product, all fp64
    from scipy.special import logsumexp, softmax

    from exact_attention_32_gb300 import WORKLOADS, workload_inputs

    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)
    b, h = head
    qs, ks, vs = (t[b:b + 1, h:h + 1].contiguous() for t in (q, k, v))
    o, lse = oracle.attention(qs, ks, vs, w.scale, w.causal)
    qd, kd, vd = (t[0, 0].double().numpy() for t in (qs, ks, vs))
    s = float(np.float32(w.scale)) * (qd @ kd.T)
    if w.causal:
        s = np.where(np.tril(np.ones_like(s, dtype=bool)), s, -np.inf)
    o_lib = softmax(s, axis=1) @ vd
    lse_lib = logsumexp(s, axis=1)
    assert np.allclose(o[0, 0], o_lib, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse[0, 0], lse_lib, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- probabilities

def test_probs_worked_example():
    # scores [2, 1, 0] (q = 1, scale 1): P = e^s / sum e^s, and P . values is
    # the printed output
    g, q, k, v = worked_example_inputs()
    P = oracle.attention_probs(q, k, 1.0, False, rows=[0])[0]
    e = np.exp(np.asarray(g["scores"]))
    assert np.allclose(P, e / e.sum(), rtol=0, atol=1e-15)
    assert abs(P @ np.asarray(g["values"]) - g["output"][0]) <= 0.5 * 10 ** -int(g["digits"][0])


@pytest.mark.parametrize("causal", [False, True])
def test_probs_times_v_is_the_dense_output(causal):
    q, k, v = make_inputs(2, 3, 77, 64, seed=61, q_gain=3.0)
    rows = np.arange(2 * 3 * 77)
    P = oracle.attention_probs(q, k, 0.125, causal, rows)
    assert np.allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    if causal:
        i = rows % 77
        assert all((P[n, i[n] + 1:] == 0).all() for n in range(rows.size))
    o_ref, _ = oracle.attention(q, k, v, 0.125, causal)
    vd = v.double().numpy().reshape(6, 77, 64)
    o = np.stack([P[n] @ vd[n // 77] for n in range(rows.size)])
    assert np.abs(o - o_ref.reshape(-1, 64)).max() < 1e-12


def test_probs_match_library_softmax():
    from scipy.special import softmax
    q, k, _ = make_inputs(1, 2, 50, 128, seed=62)
    P = oracle.attention_probs(q, k, 0.0883883461356163, False, rows=[0, 49, 50, 99])
    qd, kd = q.double().numpy(), k.double().numpy()
    for n, (h, i) in enumerate([(0, 0), (0, 49), (1, 0), (1, 49)]):
        ref = softmax(0.0883883461356163 * (qd[0, h, i] @ kd[0, h].T))
        assert np.abs(P[n] - ref).max() < 1e-15
