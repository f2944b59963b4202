"""How the E4M3 forward's error bounds in test_fp8.py were derived (not a test).

A CPU model of the E4M3 forward's rounding, in fp64: per 128-key tile the
reference max m_ref is kept until the row max has grown by more than 2^8 (in
base 2), P = 2^(s c - m_ref c) is rounded to E4M3, u and the sum of the rounded
P are scaled by 2^((m_old - m_new) c) when m_ref moves, and O = u / sum is
rounded to bf16.  Compared with exact softmax attention on the dequantised
inputs it gives the error that rounding alone causes; the bounds in
test_fp8.py are about twice the largest error it reports for each case.

    python tests/fp8_tolerance_sim.py
"""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from exact_attention_32_gb300.workloads import make_inputs, quantize_e4m3  # noqa: E402

LOG2E = 1.4426950408889634
TILE, TAU = 128, 8.0


def rounding_error(B, H, N, d, causal, q_gain, seed):
    q, k, v = make_inputs(B, H, N, d, seed=seed, q_gain=q_gain)
    (_, _, qd), (_, _, kd), (_, _, vd) = (quantize_e4m3(t) for t in (q, k, v))
    scale = float(np.float32(1 / np.sqrt(d)))
    c = scale * LOG2E
    emax, esum, n = 0.0, 0.0, 0
    for b in range(B):
        s = qd[b].double() @ kd[b].double().transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
        p = torch.exp(scale * (s - s.amax(-1, keepdim=True)))
        o_exact = (p @ vd[b].double()) / p.sum(-1, keepdim=True)
        m_ref = torch.full((H, N, 1), float("-inf"), dtype=torch.float64)
        u = torch.zeros((H, N, d), dtype=torch.float64)
        den = torch.zeros((H, N, 1), dtype=torch.float64)
        for j0 in range(0, N, TILE):
            st = s[:, :, j0:j0 + TILE]
            m_new = torch.maximum(m_ref, st.amax(-1, keepdim=True))
            need = ((m_new - m_ref) * c > TAU) | (torch.isinf(m_ref) & ~torch.isinf(m_new))
            alpha = torch.nan_to_num(torch.where(need, torch.exp2((m_ref - m_new) * c), torch.ones_like(m_ref)),
                                     nan=1.0)
            m_ref = torch.where(need, m_new, m_ref)
            mc = torch.where(torch.isinf(m_ref), torch.zeros_like(m_ref), m_ref) * c
            p8 = torch.exp2(st * c - mc).float().to(torch.float8_e4m3fn).double()
            u = u * alpha + p8 @ vd[b, :, j0:j0 + TILE].double()
            den = den * alpha + p8.sum(-1, keepdim=True)
        e = ((u / den).float().to(torch.bfloat16).double() - o_exact).abs()
        emax, esum, n = max(emax, e.max().item()), esum + e.sum().item(), n + e.numel()
    return emax, esum / n


if __name__ == "__main__":
    for causal in (False, True):
        print("large-logit 16x16x1000x128, causal", causal,
              rounding_error(16, 16, 1000, 128, causal, 8.0, 4200 + causal))
    print("large-logit 1x4x1000x128 causal", rounding_error(1, 4, 1000, 128, True, 8.0, 4100))
