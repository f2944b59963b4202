"""E4M3 forward (fa_fwd_fp8) against the fp64 oracle.

Inputs are the seeded bf16 workloads encoded per (b, h) with power-of-two
scales (exact dequantisation), so the oracle runs on exactly the values the
kernel multiplies.  The one approximation left is P rounded to E4M3 for the
P V product, and the tolerance is derived from that format alone, per output
element, from the oracle's fp64 weights P and the values V.

Rounding.  E4M3 keeps 3 mantissa bits: rounding a normal value (>= 2^-6)
to nearest moves it by at most 2^-4 of itself; below 2^-6 the step is 2^-9,
so a subnormal moves by at most min(2^-10, itself).  The kernel's
exponentials are relative to a reference at or below the row max, so its
largest term is >= 1 and its terms are at least the weights scaled by
1 / max P.  In weight units the error of key j is therefore at most
e_j = P_j 2^-4 if P_j >= 2^-6 max P, else min(P_j, 2^-10 max P).

Propagation.  O = sum_j p^_j v_j / L.  Dividing by the sum of the rounded
terms, O' - O = sum_j (p^_j - p_j)(v_j - O) / L; dividing by the fp32 sum
of the unrounded terms, a key contributes (p^_j - p_j) v_j instead.
fa_fwd_fp8 divides by the rounded sum in every tile where one key can carry a
quarter of the row (its documented contract), so keys with P_j > 1/4 take
dev_jc = |v_jc - O_c|, and every other key dev_jc = |v_jc| + |O_c| (which is
>= both forms).

* Worst case, every element: |dO_c| <= sum_j e_j dev_jc / (1 - sum_j e_j),
  plus 2^-8 |O_c| for the bf16 output and 1e-5 for fp32 arithmetic.
* Typical case, the mean over all checked elements: the rounding errors of
  different keys are independent with mean zero.  A normal value placed at
  random within its binade (density ~ 1/x) has relative rounding variance
  c^2 = (2^-3)^2 / 12 * 3 / (8 ln 2); a subnormal has variance (2^-9)^2 / 12
  in units of max P (at most P_j^2).  With s_jc^2 = var_j dev_jc^2 the error
  of an element is about normal with standard deviation sqrt(sum_j s_jc^2), so
  its expected magnitude is sqrt(2/pi) times that, plus 2^-10 |O_c| for the
  output rounding.  The measured mean must stay within 1.25 times the mean of
  that expectation.
LSE is computed from the unrounded fp32 sum: max |dLSE| <= 1e-3 as for bf16.
A CPU test checks both on a simulation of the rounding (any reference offset,
any choice of divisor outside the heavy keys) and that they catch a coarser
format and a wrong divisor.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_32_gb300 import WORKLOADS, make_inputs, workload_inputs
from exact_attention_32_gb300.workloads import quantize_e4m3, sample_rows

MAX_LSE = 1e-3
E4M3_REL, E4M3_MIN_NORMAL, E4M3_SUB_HALF = 2.0 ** -4, 2.0 ** -6, 2.0 ** -10
REL_VAR = (2.0 ** -3) ** 2 / 12 * 3 / (8 * math.log(2))
SUB_VAR = (2.0 ** -9) ** 2 / 12
BF16_REL = 2.0 ** -8
HEAVY = 0.25 * (1 + 1e-3)  # keys above a quarter of the row (with a margin for the kernel's fp32 sums)
MEAN_SLACK = 1.25


def e4m3_bounds(P, V, O):
    """Per-element worst-case bound and expected magnitude of |dO| for rows of
    one (b, h) slice: weights P [R, N], the slice's values V [N, d], exact
    outputs O [R, d]."""
    pmax = P.max(axis=1, keepdims=True)
    normal = P >= E4M3_MIN_NORMAL * pmax
    e = np.where(normal, E4M3_REL * P, np.minimum(P, E4M3_SUB_HALF * pmax))
    var = np.where(normal, REL_VAR * P ** 2, np.minimum(P ** 2, SUB_VAR * pmax ** 2))
    heavy = P > HEAVY
    el, vl = np.where(heavy, 0.0, e), np.where(heavy, 0.0, var)
    aV, aO = np.abs(V), np.abs(O)
    # light keys: dev = |v| + |O|; heavy keys (at most three per row): |v - O|
    num = el @ aV + aO * el.sum(axis=1, keepdims=True)
    sq = vl @ (V ** 2) + 2 * aO * (vl @ aV) + aO ** 2 * vl.sum(axis=1, keepdims=True)
    r, j = np.nonzero(heavy)
    dv = np.abs(V[j] - O[r])
    np.add.at(num, r, e[r, j][:, None] * dv)
    np.add.at(sq, r, var[r, j][:, None] * dv ** 2)
    w = num / (1.0 - e.sum(axis=1, keepdims=True))
    worst = w + BF16_REL * (aO + w) + 1e-5
    typical = math.sqrt(2 / math.pi) * np.sqrt(sq) + 0.25 * BF16_REL * aO
    return worst, typical


def check_against_bounds(o, lse, o_ref, lse_ref, worst, typical):
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    e, le = np.abs(o - o_ref), np.abs(lse - lse_ref)
    log = os.environ.get("FA_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "max_dO": float(e.max()), "mean_dO": float(e.mean()),
                                "max_dO_over_bound": float((e / worst).max()),
                                "mean_dO_over_expected": float(e.mean() / typical.mean()),
                                "max_dLSE": float(le.max())}) + "\n")
    assert (e <= worst).all(), f"max |dO| / bound = {(e / worst).max():.3f}"
    assert e.mean() <= MEAN_SLACK * typical.mean(), (e.mean(), typical.mean())
    assert le.max() <= MAX_LSE, le.max()


def bounds_for_rows(qd, kd, vd, scale, causal, rows, o_ref):
    """The bounds of flat rows ``rows`` (sorted) of the dequantised inputs,
    computed slice by slice."""
    B, H, N, d = qd.shape
    rows = np.asarray(rows)
    vv = vd.double().numpy().reshape(B * H, N, d)
    worst, typical = np.empty_like(o_ref), np.empty_like(o_ref)
    bh_of = rows // N
    for bh in np.unique(bh_of):
        sel = np.nonzero(bh_of == bh)[0]
        b, h = divmod(int(bh), H)
        one = slice(b, b + 1), slice(h, h + 1)
        P = oracle.attention_probs(qd[one], kd[one], scale, causal, rows[sel] - bh * N)
        worst[sel], typical[sel] = e4m3_bounds(P, vv[bh], o_ref[sel])
    return worst, typical


# ------------------------------------------------------------ CPU: the bound

def simulate_e4m3_rounding(P, V, rng, heavy_rule=True, fmt=torch.float8_e4m3fn):
    """O computed from weights P [R, N] rounded to an 8-bit format, relative
    to a random reference 0..8 octaves below each row's max, divided by the
    rounded sum for the heavy keys (if heavy_rule) and a random half of the
    others, and by the unrounded sum for the rest.  V [N, d]."""
    p = P / P.max(axis=1, keepdims=True) * 2.0 ** rng.uniform(0, 8, size=(P.shape[0], 1))
    pr = torch.from_numpy(p).float().to(fmt).double().numpy()
    rounded = rng.random(p.shape) < 0.5
    if heavy_rule:
        rounded |= P > 0.25
    L = (pr * rounded).sum(axis=1, keepdims=True) + (p * ~rounded).sum(axis=1, keepdims=True)
    return (pr @ V) / L


@pytest.mark.parametrize("q_gain,causal", [(1.0, False), (1.0, True), (8.0, True), (8.0, False)])
def test_bound_holds_on_simulated_rounding(q_gain, causal):
    N = 1000
    q, k, v = make_inputs(1, 1, N, 128, seed=4300 + int(q_gain) + causal, q_gain=q_gain)
    P = oracle.attention_probs(q, k, 0.0883883461356163, causal, np.arange(N))
    V = v.double().numpy()[0, 0]
    O = P @ V
    worst, typical = e4m3_bounds(P, V, O)
    rng = np.random.default_rng(1)
    for _ in range(3):
        e = np.abs(simulate_e4m3_rounding(P, V, rng) - O)
        assert (e <= worst).all()
        assert e.mean() <= typical.mean() and e.mean() >= 0.5 * typical.mean()
    # the bounds are not vacuous: a coarser format (E5M2, half-step 2^-3)
    # breaks the expected magnitude, and dividing every key by the unrounded
    # sum breaks the worst case on rows that one key carries
    e = np.abs(simulate_e4m3_rounding(P, V, rng, fmt=torch.float8_e5m2) - O)
    assert e.mean() > MEAN_SLACK * typical.mean()
    if q_gain > 1:
        p = P / P.max(axis=1, keepdims=True)
        sim = (torch.from_numpy(p).float().to(torch.float8_e4m3fn).double().numpy() @ V) / p.sum(1, keepdims=True)
        assert (np.abs(sim - O) > worst).any()


def test_quantization_is_exact_in_bf16():
    q, _, _ = make_inputs(2, 3, 100, 128, seed=1, q_gain=8.0)
    q8, s, deq = quantize_e4m3(q)
    assert q8.dtype == torch.float8_e4m3fn and s.shape == (2, 3)
    assert torch.all(torch.log2(s) == torch.round(torch.log2(s)))
    assert torch.equal(deq.double(), q8.double() * s.double()[..., None, None])
    assert (q8.float().abs().amax(dim=(-1, -2)) <= 448).all()


def run(q, k, v, scale, causal):
    from exact_attention_32_gb300 import fa_get_device_status, forward_fp8
    (q8, qs, qd), (k8, ks, kd), (v8, vs, vd) = (quantize_e4m3(t) for t in (q, k, v))
    o, lse = forward_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qs.cuda(), ks.cuda(), vs.cuda(), scale=scale,
                         causal=causal)
    torch.cuda.synchronize()
    assert fa_get_device_status(0) == 0
    return o.double().cpu().numpy(), lse.double().cpu().numpy(), (qd, kd, vd)


def check_rows(o, lse, deq, scale, causal, rows=None):
    """Compare rows (all when None) of the kernel's output with the oracle on
    the dequantised inputs, against the E4M3 bounds of those rows."""
    qd, kd, vd = deq
    B, H, N, d = qd.shape
    if rows is None:
        rows = np.arange(B * H * N)
    o_ref, lse_ref = oracle.attention(qd, kd, vd, scale, causal, rows=rows)
    worst, typical = bounds_for_rows(qd, kd, vd, scale, causal, rows, o_ref)
    check_against_bounds(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, worst, typical)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 127, 128, 129, 256, 300, 1000])
def test_small_problems_every_row(N, causal):
    q, k, v = make_inputs(2, 2, N, 128, seed=4000 + N + causal)
    scale = float(np.float32(1 / np.sqrt(128)))
    o, lse, deq = run(q, k, v, scale, causal)
    check_rows(o, lse, deq, scale, causal)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["b4_h16_n2048_d128", "b2_h32_n4096_d128_causal", "b1_h32_n16384_d128_causal"])
def test_workloads_sampled_rows(name):
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)
    o, lse, deq = run(q, k, v, w.scale, w.causal)
    rows = sample_rows(w.B, w.H, w.N, per_head=16, seed=w.seed)
    check_rows(o, lse, deq, w.scale, w.causal, rows)


@pytest.mark.gpu
def test_large_logits():
    q, k, v = make_inputs(1, 4, 1000, 128, seed=4100, q_gain=8.0)
    o, lse, deq = run(q, k, v, 0.0883883461356163, True)
    check_rows(o, lse, deq, 0.0883883461356163, True)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_large_logits_every_row(causal):
    # many rows carried by one or two keys, where the E4M3 rounding of P and the
    # divisor of O matter most
    q, k, v = make_inputs(16, 16, 1000, 128, seed=4200 + causal, q_gain=8.0)
    scale = float(np.float32(1 / np.sqrt(128)))
    o, lse, deq = run(q, k, v, scale, causal)
    check_rows(o, lse, deq, scale, causal)


@pytest.mark.gpu
def test_head_dim_64_unsupported():
    import exact_attention_32_gb300 as fa
    q8 = torch.zeros((1, 1, 128, 64), dtype=torch.uint8, device="cuda")
    s = torch.ones(1, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.forward_fp8(q8, q8, q8, s, s, s)
    assert e.value.status == 2
