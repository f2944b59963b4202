"""GPU parity of the backward (fa_bwd) against the fp64 oracle.

The GPU gets Q, K, V, dO and its own forward's O and LSE; the oracle
recomputes everything from Q, K, V, dO.  Tolerances, per gradient G
(bf16 inputs, P and dS rounded to bf16 for the MMAs, bf16 outputs):
    max |G - G_ref| <= 2e-2 * max |G_ref|,   mean |G - G_ref| <= 1e-2 * mean |G_ref|.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_32_gb300 import (WORKLOADS, backward, fa_get_device_status, forward, make_inputs,
                                      workload_inputs)
from exact_attention_32_gb300.workloads import make_grad_output

pytestmark = pytest.mark.gpu
REL_MAX, REL_MEAN = 2e-2, 1e-2


def gpu_grads(q, k, v, do, scale, causal):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = forward(qd, kd, vd, scale=scale, causal=causal)
    dq, dk, dv = backward(qd, kd, vd, o, lse, dod, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa_get_device_status(0) == 0
    return {n: t.double().cpu().numpy() for n, t in (("dq", dq), ("dk", dk), ("dv", dv))}


def check(got, ref, slices=None):
    B, H, N, d = got["dq"].shape
    out = {}
    # a gradient that is zero by construction (dQ at N = 1) is compared on the
    # scale of the problem's largest gradient: the GPU's dP and D are summed in
    # different orders, so dP - D is a rounding residual, not an exact zero
    floor = 1e-3 * max(np.abs(ref[n]).max() for n in ("dq", "dk", "dv"))
    for name in ("dq", "dk", "dv"):
        g = got[name].reshape(B * H, N, d)
        if slices is not None:
            g = g[slices]
        r = ref[name]
        assert np.isfinite(g).all(), name
        err = np.abs(g - r)
        scale_max, scale_mean = max(np.abs(r).max(), floor), max(np.abs(r).mean(), floor)
        out[name] = (float(err.max() / max(scale_max, 1e-30)), float(err.mean() / max(scale_mean, 1e-30)))
        log = os.environ.get("FA_PARITY_LOG")
        if log:
            with open(log, "a") as f:
                f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                    "grad": name, "rel_max": out[name][0], "rel_mean": out[name][1]}) + "\n")
        assert err.max() <= REL_MAX * scale_max, (name, out[name])
        assert err.mean() <= REL_MEAN * scale_mean, (name, out[name])
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 64, 128, 129, 255, 256, 300, 1000])
def test_small_problems_all_rows(N, d, causal):
    q, k, v = make_inputs(2, 2, N, d, seed=3000 + N + d + causal)
    do = make_grad_output(2, 2, N, d, seed=3000 + N)
    scale = float(np.float32(1 / np.sqrt(d)))
    got = gpu_grads(q, k, v, do, scale, causal)
    ref = oracle.attention_backward(q, k, v, do, scale, causal)
    check(got, ref)


@pytest.mark.parametrize("name,slices", [("b1_h1_n256_d64", None),
                                         ("b16_h16_n1000_d64_causal_q8", [0, 17, 100, 255]),
                                         ("b4_h16_n2048_d128", [0, 33, 63]),
                                         ("b2_h32_n4096_d128_causal", [0, 63]),
                                         ("b1_h32_n16384_d128_causal", [5])])
def test_workloads(name, slices):
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)
    do = make_grad_output(w.B, w.H, w.N, w.d, seed=w.seed)
    got = gpu_grads(q, k, v, do, w.scale, w.causal)
    ref = oracle.attention_backward(q, k, v, do, w.scale, w.causal, slices=slices)
    check(got, ref, slices)


def test_many_key_blocks_per_sm():
    # 8 x 64 slices of 300 rows: 1536 key-block CTAs, several waves
    q, k, v = make_inputs(8, 64, 300, 64, seed=31)
    do = make_grad_output(8, 64, 300, 64, seed=31)
    got = gpu_grads(q, k, v, do, 0.125, True)
    ref = oracle.attention_backward(q, k, v, do, 0.125, True, slices=[0, 1, 200, 511])
    check(got, ref, [0, 1, 200, 511])


def test_deterministic_dk_dv():
    q, k, v = (t.cuda() for t in make_inputs(1, 4, 500, 128, seed=32))
    do = make_grad_output(1, 4, 500, 128, seed=32, device="cuda")
    o, lse = forward(q, k, v, causal=True)
    a = backward(q, k, v, o, lse, do, causal=True)
    b = backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    # dK, dV are accumulated in one CTA in a fixed order: bit-identical
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dQ sums partials from several CTAs with atomics: equal up to rounding order
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2 ** -6 * a[0].float().abs().max().item()


@pytest.mark.parametrize("d,causal", [(64, True), (128, False)])
def test_autograd_attention(d, causal):
    # attention() through torch.autograd: the loss sum(O * dO) backpropagates
    # through fa_bwd to the oracle's gradients, and to the direct calls' dK and dV
    # bit for bit (dQ is summed by reductions in L2, in no fixed order)
    import exact_attention_32_gb300 as fa
    q, k, v = make_inputs(1, 3, 300, d, seed=4100 + d)
    do = make_grad_output(1, 3, 300, d, seed=4100 + d)
    scale = float(np.float32(1 / np.sqrt(d)))
    qd, kd, vd = (t.cuda().requires_grad_(True) for t in (q, k, v))
    o = fa.attention(qd, kd, vd, scale=scale, causal=causal)
    (o.float() * do.cuda().float()).sum().backward()
    torch.cuda.synchronize()
    got = {"dq": qd.grad.double().cpu().numpy(), "dk": kd.grad.double().cpu().numpy(),
           "dv": vd.grad.double().cpu().numpy()}
    check(got, oracle.attention_backward(q, k, v, do, scale, causal))
    direct = gpu_grads(q, k, v, do, scale, causal)
    for name in ("dk", "dv"):
        assert np.array_equal(got[name], direct[name]), name
    assert np.abs(got["dq"] - direct["dq"]).max() <= 1e-2 * np.abs(direct["dq"]).max()
