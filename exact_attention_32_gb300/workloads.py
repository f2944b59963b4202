"""Seeded synthetic workloads for exact attention forward.

This module only names problem sizes and draws random inputs.  It holds none of
the attention arithmetic, so both the CUDA path's tests/benchmark and the
oracle can be fed from it.

Every workload is self-attention over contiguous [B, H, N, d] bf16 tensors
(the layout of "6.1 FlashAttention V1 in detail", section 8.1).  Inputs are
drawn iid N(0, 1) in fp32 from a CPU ``torch.Generator`` in the order Q, K, V,
Q is multiplied by ``q_gain`` (8 for the large-logit stress case; a power of two,
so it commutes with the bf16 rounding that follows), and all three are rounded
to bf16 (round-to-nearest-even).  The softmax scale is the fp32 value of
1/sqrt(d), the value the kernels receive.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    q_gain: float
    seed: int

    @property
    def scale(self) -> float:
        """fp32 value of 1/sqrt(d), returned as a Python float."""
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def flops(self) -> float:
        """Conventional forward FLOPs: 4*B*H*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def min_bytes(self) -> int:
        """Algorithmic minimum HBM traffic: read Q, K, V once, write O (bf16) and LSE (fp32)."""
        return self.B * self.H * self.N * (4 * self.d * 2 + 4)

    def shape(self):
        return (self.B, self.H, self.N, self.d)


WORKLOADS = {w.name: w for w in [
    Workload("b1_h1_n256_d64", 1, 1, 256, 64, False, 1.0, 1001),
    Workload("b4_h16_n2048_d128", 4, 16, 2048, 128, False, 1.0, 1002),
    Workload("b16_h16_n1000_d64_causal_q8", 16, 16, 1000, 64, True, 8.0, 1003),
    Workload("b2_h32_n4096_d128_causal", 2, 32, 4096, 128, True, 1.0, 1004),
    Workload("b1_h32_n16384_d128_causal", 1, 32, 16384, 128, True, 1.0, 1005),
    Workload("b1_h32_n16384_d128", 1, 32, 16384, 128, False, 1.0, 1005),
]}

# the long-sequence causal run that the throughput target is quoted on
HEADLINE = "b1_h32_n16384_d128_causal"


def make_inputs(B: int, H: int, N: int, d: int, seed: int, q_gain: float = 1.0,
                device="cpu"):
    """Draw (q, k, v) bf16 [B, H, N, d] from ``seed`` (CPU generator, fp32
    N(0,1) in the order Q, K, V; Q *= q_gain; round to bf16), then move them
    to ``device``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if q_gain != 1.0:
        q.mul_(q_gain)
    out = []
    for t in (q, k, v):
        t = t.to(torch.bfloat16)
        out.append(t.to(device) if str(device) != "cpu" else t)
    return tuple(out)


def make_grad_output(B: int, H: int, N: int, d: int, seed: int, device="cpu"):
    """A seeded upstream gradient dO for the backward: iid N(0,1) fp32 from a
    CPU generator seeded with ``seed + 7919``, rounded to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    t = torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return t.to(device) if str(device) != "cpu" else t


def quantize_e4m3(t: torch.Tensor):
    """Encode a [B, H, N, d] tensor as E4M3 with one power-of-two fp32 scale per
    (b, h): scale = 2^ceil(log2(absmax / 448)), t8 = round_to_e4m3(t / scale).
    Returns (t8 float8_e4m3fn, scale fp32 [B, H], dequantised bf16 t8 * scale).
    With a power-of-two scale the dequantised values are exact in bf16."""
    a = t.float().abs().amax(dim=(-1, -2))
    a = torch.where(a > 0, a, torch.ones_like(a))
    scale = torch.exp2(torch.ceil(torch.log2(a / 448.0)))
    t8 = (t.float() / scale[..., None, None]).to(torch.float8_e4m3fn)
    deq = (t8.float() * scale[..., None, None]).to(torch.bfloat16)
    return t8, scale.contiguous(), deq


def workload_inputs(w: Workload, device="cpu", seed=None):
    """Inputs of a named workload (its own seed unless one is given)."""
    return make_inputs(w.B, w.H, w.N, w.d, w.seed if seed is None else seed,
                       w.q_gain, device)


def sample_rows(B: int, H: int, N: int, per_head: int, seed: int, tile: int = 128):
    """Flat row ids (b*H + h)*N + i for spot checks at full size: in every
    (b, h) slice the first and last rows, the rows on both sides of every
    ``tile`` boundary (up to ``per_head`` of them) and random rows to fill
    ``per_head``.  Sorted, unique."""
    rng = np.random.default_rng(seed)
    fixed = {0, N - 1}
    for t in range(tile, N, tile):
        fixed.update((t - 1, t))
    fixed = sorted(i for i in fixed if 0 <= i < N)
    if len(fixed) > per_head:
        pick = np.linspace(0, len(fixed) - 1, per_head).round().astype(int)
        fixed = [fixed[p] for p in pick]
    rest = np.setdiff1d(np.arange(N), np.asarray(fixed, dtype=np.int64))
    rows = []
    for bh in range(B * H):
        extra = min(per_head - len(fixed), rest.size)
        rnd = rng.choice(rest, size=extra, replace=False) if extra > 0 else []
        idx = sorted(set(fixed) | set(int(x) for x in rnd))
        rows.extend(bh * N + i for i in idx)
    return np.asarray(rows, dtype=np.int64)
