"""Exact-attention oracle: plain, slow, obviously correct CPU references.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (and its ``--impl reference`` arm) may import this
package.  It shares no code with the CUDA path and never calls it; the CUDA
path never calls it either.

Independent references, each in fp64 or better:

``attention``          the plain definition ("6.1 FlashAttention V1 in detail",
                       section 1.1: S = scale * Q K^T, P = softmax(S), O = P V)
                       with the softmax written as the three-pass safe softmax of
                       section 3.1 and LSE = m + log(l) ("FlashAttention:
                       IO-Aware Tiling, ...", section "Backward Pass
                       Recomputation").  Compiled C (``attn_oracle.c``), OpenMP
                       over rows, so that full-size rows stay affordable.
``attention_online``   the tile-by-tile (m, l, u) merge of "FlashAttention:
                       optimize data movement before counting FLOPs", section 02
                       (m' = max(m, max s); l' = e^(m-m') l + sum e^(s-m');
                       u' = e^(m-m') u + sum e^(s-m') V; output u'/l'), in numpy
                       fp64, with any tile sizes and any K/V-tile visiting order.
                       It exists to pin the online reasoning, not the GPU.
``merge``              the two-block merge of "FlashAttention: IO-Aware Tiling,
                       ...", section "Online Softmax Mathematics", folding
                       partial (O, LSE) results over disjoint key ranges.
``attention_backward`` gradients dQ, dK, dV of sum(O * dO), in numpy fp64, by
                       the formulas of "6.1 FlashAttention V1 in detail",
                       section 6.1 (dV = P^T dO, dP = dO V^T, D = rowsum(dO * O)
                       = rowsum(dP * P), dS = P * (dP - D)) and of the
                       llms.blog page, section "Backward Pass Recomputation"
                       (dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d), with 1/sqrt(d)
                       read as the scale), dense per (b, h) slice.
``attention_blocksparse`` the plain definition with a 0/1 block mask over
                       (query block, key block) pairs: keys of a masked block
                       take no part for the rows of that query block (numpy fp64,
                       dense per slice).
``attention_probs``    the softmax weights P themselves (numpy fp64, plain
                       definition, for selected rows): what the E4M3 forward's
                       error bound is computed from.
``attention_decimal``  brute force in Python ``decimal`` at 50 digits, using
                       the softmax definition directly (exp(s_j) / sum exp(s_k),
                       no max shift) - an independent formulation for tiny
                       inputs.

Readings where the pages are silent (shared by all three):
  * ``scale`` is applied exactly as given (the configs use 1/sqrt(d), passed
    as the fp32 value the GPU receives);
  * causal keeps keys j <= i for query row i (N_q = N_k);
  * the log is natural, over the scaled logits.

Every function here is pinned by ``tests/test_oracle.py`` against values the
pages print, closed forms, invariants and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from decimal import Decimal, getcontext

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, OpenMP
    when available, never -ffast-math).  Returns the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_double, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int64, ctypes.c_int64]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the compiled oracle uses by default."""
    return int(_load().oracle_max_threads())


def _bf16_bits(t) -> np.ndarray:
    """bf16 torch tensor (CPU) -> contiguous uint16 numpy view of its bits."""
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError("oracle inputs are bf16 tensors")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _as_f64(t) -> np.ndarray:
    """bf16 torch tensor -> float64 numpy array (exact widening)."""
    import torch
    return t.detach().cpu().to(torch.float64).numpy()


def attention(q, k, v, scale: float, causal: bool, rows=None, threads: int = 0, kv_range=None):
    """fp64 attention of bf16 inputs by the plain definition.

    q, k, v  : bf16 CPU tensors [B, H, N, d]
    rows     : None (all rows) or an int64 array of flat row ids
               (b*H + h)*N + i
    kv_range : None (all keys) or (lo, hi): only keys lo <= j < hi take part;
               a row that then admits no key gets O = 0, LSE = -inf
    Returns (O, LSE) as float64 numpy arrays: [B, H, N, d] and [B, H, N] for
    all rows, else [len(rows), d] and [len(rows)].
    """
    B, H, N, d = q.shape
    if tuple(k.shape) != (B, H, N, d) or tuple(v.shape) != (B, H, N, d):
        raise ValueError("q, k, v must share the shape [B, H, N, d]")
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    if rows is None:
        n_rows = B * H * N
        rows_arr = None
        rows_ptr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.size
        rows_ptr = rows_arr.ctypes.data
    o = np.empty((n_rows, d), dtype=np.float64)
    lse = np.empty((n_rows,), dtype=np.float64)
    lo, hi = (0, N) if kv_range is None else (int(kv_range[0]), int(kv_range[1]))
    rc = _load().oracle_attention_rows(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, B, H, N, d,
        float(scale), int(bool(causal)), rows_ptr, n_rows,
        o.ctypes.data, lse.ctypes.data, int(threads), lo, hi)
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed ({rc})")
    if rows is None:
        return o.reshape(B, H, N, d), lse.reshape(B, H, N)
    return o, lse


def attention_online(q, k, v, scale: float, causal: bool, block_q: int,
                     block_k: int, order=None, mask_tail: bool = True):
    """Tile-by-tile online softmax with the (m, l, u) merge, fp64 numpy.

    Q is cut into tiles of ``block_q`` rows and K/V into tiles of ``block_k``
    rows (the last tiles may be partial); each Q tile visits the K/V tiles in
    ``order`` (a permutation of range(T_c); default ascending).  Per visit:
        s  = scale * Q_i K_j^T       (columns past N, and causal j > i, -> -inf)
        m' = max(m, rowmax s)
        l' = exp(m - m') l + rowsum exp(s - m')
        u' = exp(m - m') u + exp(s - m') V_j
    and finally O = u / l, LSE = m + log l.  A row whose m' is still -inf (every
    key seen so far masked) keeps m = -inf, l = 0, u = 0.

    ``mask_tail=False`` pads the last K/V tile with zero rows and lets their
    scores (0) into the softmax - the mistake the K/V out-of-range mask exists
    to prevent ("6.1 FlashAttention V1 in detail", section 8.3).  It is here
    only so a test can show that the mistake is caught.
    """
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = qd.shape
    t_c = -(-N // block_k)
    if order is None:
        order = range(t_c)
    order = list(order)
    if sorted(order) != list(range(t_c)):
        raise ValueError("order must be a permutation of the K/V tiles")
    pad = t_c * block_k - N
    kp = np.concatenate([kd, np.zeros((B, H, pad, d))], axis=2) if pad else kd
    vp = np.concatenate([vd, np.zeros((B, H, pad, d))], axis=2) if pad else vd
    o = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    for i0 in range(0, N, block_q):
        i1 = min(i0 + block_q, N)
        qi = qd[:, :, i0:i1, :]
        rows = np.arange(i0, i1)
        m = np.full((B, H, i1 - i0), -np.inf)
        l = np.zeros((B, H, i1 - i0))
        u = np.zeros((B, H, i1 - i0, d))
        for j in order:
            j0, j1 = j * block_k, (j + 1) * block_k
            s = scale * np.einsum("bhic,bhjc->bhij", qi, kp[:, :, j0:j1, :])
            cols = np.arange(j0, j1)
            if mask_tail:
                s[..., cols >= N] = -np.inf
            if causal:
                s[..., cols[None, :] > rows[:, None]] = -np.inf
            m_new = np.maximum(m, s.max(axis=-1))
            live = np.isfinite(m_new)
            ref = np.where(live, m_new, 0.0)
            alpha = np.where(live, np.exp(m - ref), 1.0)
            p = np.exp(s - ref[..., None])
            l = alpha * l + p.sum(axis=-1)
            u = alpha[..., None] * u + np.einsum("bhij,bhjc->bhic", p, vp[:, :, j0:j1, :])
            m = m_new
        o[:, :, i0:i1, :] = u / l[..., None]
        lse[:, :, i0:i1] = m + np.log(l)
    return o, lse


def merge(o_parts, lse_parts):
    """Merge partial attention results over disjoint key ranges, fp64.

    o_parts [S, ..., d] (each normalised over its own keys) and lse_parts
    [S, ...] (each m_s + ln l_s).  The parts are folded in one at a time with
    the two-block merge of "FlashAttention: IO-Aware Tiling, ...", section
    "Online Softmax Mathematics", taking each part as (m_s, l_s, O_s) with
    m_s = LSE_s and l_s = 1:
        m = max(m1, m2),  l = e^(m1-m) l1 + e^(m2-m) l2,
        O = (l1 e^(m1-m) / l) O1 + (l2 e^(m2-m) / l) O2.
    A part with LSE = -inf (no admitted key) carries no weight.  Returns
    (O, LSE = m + ln l).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.full(lse_parts.shape[1:], -np.inf)
    l = np.zeros(lse_parts.shape[1:])
    o = np.zeros(o_parts.shape[1:])
    for s in range(lse_parts.shape[0]):
        m2, l2, o2 = lse_parts[s], np.where(np.isfinite(lse_parts[s]), 1.0, 0.0), o_parts[s]
        m_new = np.maximum(m, m2)
        ref = np.where(np.isfinite(m_new), m_new, 0.0)
        a1 = np.where(l > 0, l * np.exp(m - ref), 0.0)
        a2 = np.where(l2 > 0, l2 * np.exp(m2 - ref), 0.0)
        l_new = a1 + a2
        with np.errstate(invalid="ignore", divide="ignore"):
            o = np.where((l_new > 0)[..., None],
                         (a1 / l_new)[..., None] * o + (a2 / l_new)[..., None] * o2, 0.0)
        m, l = m_new, l_new
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse


def attention_backward(q, k, v, do, scale: float, causal: bool, slices=None):
    """fp64 gradients of sum(O * dO) with respect to Q, K and V.

    q, k, v, do : bf16 CPU tensors [B, H, N, d] (widened exactly)
    slices      : None (all) or an iterable of flat slice ids b*H + h
    Per slice, dense: S = scale Q K^T (causal: -inf above the diagonal),
    P by the three-pass safe softmax, O = P V; then dV = P^T dO,
    dP = dO V^T, D_i = rowsum(dO * O)_i, dS = P * (dP - D),
    dQ = scale dS K, dK = scale dS^T Q.
    Returns dict of float64 arrays dq, dk, dv ([n_slices, N, d]), o
    ([n_slices, N, d]), lse and D ([n_slices, N]), in the order of `slices`.
    """
    qd, kd, vd, dod = (_as_f64(t) for t in (q, k, v, do))
    B, H, N, d = qd.shape
    qd, kd, vd, dod = (x.reshape(B * H, N, d) for x in (qd, kd, vd, dod))
    ids = list(range(B * H)) if slices is None else [int(x) for x in slices]
    out = {name: [] for name in ("dq", "dk", "dv", "o", "lse", "D")}
    mask = np.triu(np.ones((N, N), dtype=bool), k=1) if causal else None
    for bh in ids:
        Q, K, V, dO = qd[bh], kd[bh], vd[bh], dod[bh]
        S = scale * (Q @ K.T)
        if causal:
            S[mask] = -np.inf
        m = S.max(axis=1, keepdims=True)          # pass 1
        E = np.exp(S - m)
        l = E.sum(axis=1, keepdims=True)          # pass 2
        P = E / l                                 # pass 3
        O = P @ V
        dV = P.T @ dO
        dP = dO @ V.T
        D = (dO * O).sum(axis=1, keepdims=True)
        dS = P * (dP - D)
        out["dq"].append(scale * (dS @ K))
        out["dk"].append(scale * (dS.T @ Q))
        out["dv"].append(dV)
        out["o"].append(O)
        out["lse"].append((m + np.log(l))[:, 0])
        out["D"].append(D[:, 0])
    return {name: np.stack(vals) for name, vals in out.items()}


def attention_blocksparse(q, k, v, scale: float, causal: bool, block_mask, block: int = 128):
    """fp64 attention restricted by a block mask ("FlashAttention: optimize data
    movement before counting FLOPs", section 07, names the block-sparse variant;
    the reading here: key j is admitted to query i only if
    block_mask[i // block][j // block] is nonzero, and, when causal, j <= i).
    Per slice: dense scores, masked entries -inf, the three-pass softmax of
    the plain definition; a row with no admitted key gets O = 0, LSE = -inf.
    block_mask: [ceil(N/block), ceil(N/block)] array, shared by all (b, h).
    Returns (O [B, H, N, d], LSE [B, H, N]) float64."""
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = qd.shape
    bm = np.asarray(block_mask).astype(bool)
    nb = -(-N // block)
    if bm.shape != (nb, nb):
        raise ValueError("block_mask must be [ceil(N/block), ceil(N/block)]")
    idx = np.arange(N) // block
    allowed = bm[idx[:, None], idx[None, :]]
    if causal:
        allowed &= np.tril(np.ones((N, N), dtype=bool))
    o = np.zeros((B, H, N, d))
    lse = np.full((B, H, N), -np.inf)
    live = allowed.any(axis=1)
    for b in range(B):
        for h in range(H):
            S = scale * (qd[b, h] @ kd[b, h].T)
            S[~allowed] = -np.inf
            Sl = S[live]
            m = Sl.max(axis=1, keepdims=True)        # pass 1
            E = np.exp(Sl - m)
            l = E.sum(axis=1, keepdims=True)         # pass 2
            o[b, h, live] = (E / l) @ vd[b, h]       # pass 3
            lse[b, h, live] = (m + np.log(l))[:, 0]
    return o, lse


def attention_probs(q, k, scale: float, causal: bool, rows):
    """The softmax weights P of the plain definition ("6.1 FlashAttention V1 in
    detail", section 1.1: S = scale * Q K^T, P = softmax(S) row-wise), fp64,
    for the flat row ids ``rows`` ((b*H + h)*N + i).  Masked keys (j > i when
    causal) get weight 0.  Returns float64 numpy [len(rows), N]."""
    qd, kd = _as_f64(q), _as_f64(k)
    B, H, N, d = qd.shape
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, N))
    bh_of, i_of = np.divmod(rows, N)
    for bh in np.unique(bh_of):
        sel = np.nonzero(bh_of == bh)[0]
        b, h = divmod(int(bh), H)
        s = scale * (qd[b, h, i_of[sel]] @ kd[b, h].T)      # scores of these rows
        if causal:
            s[np.arange(N)[None, :] > i_of[sel][:, None]] = -np.inf
        e = np.exp(s - s.max(axis=1, keepdims=True))
        out[sel] = e / e.sum(axis=1, keepdims=True)
    return out


def attention_decimal(q, k, v, scale, causal: bool, digits: int = 50):
    """Brute force in ``decimal``: softmax by its definition, no max shift.

    P_ij = exp(s_ij) / sum_k exp(s_ik) over admitted keys; O_i = sum_j P_ij V_j;
    LSE_i = ln(sum_k exp(s_ik)).  For tiny inputs only (pure Python loops).
    Returns nested lists of Decimal: O [B][H][N][d], LSE [B][H][N].
    """
    getcontext().prec = digits
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = qd.shape
    sc = Decimal(float(scale))
    O = [[[[None] * d for _ in range(N)] for _ in range(H)] for _ in range(B)]
    L = [[[None] * N for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            for i in range(N):
                keys = range(i + 1) if causal else range(N)
                e = {}
                for j in keys:
                    dot = sum(Decimal(float(qd[b, h, i, c])) * Decimal(float(kd[b, h, j, c]))
                              for c in range(d))
                    e[j] = (sc * dot).exp()
                z = sum(e.values())
                for c in range(d):
                    O[b][h][i][c] = sum(e[j] * Decimal(float(vd[b, h, j, c])) for j in keys) / z
                L[b][h][i] = z.ln()
    return O, L
