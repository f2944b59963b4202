"""ctypes binding of libfa.so: argument marshalling only.

Every function of include/fa.h is exposed under the same name; ``forward`` is
the tensor-level convenience call.  Torch supplies device memory and the
current stream; all arithmetic runs in the library's CUDA kernels.  There is
no fallback: if libfa.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")
_lib = None
_lock = threading.Lock()

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_NO_DEVICE",
                4: "FA_ERR_ARCH", 5: "FA_ERR_LAUNCH", 6: "FA_ERR_TIMEOUT", 7: "FA_ERR_WORKSPACE_LIMIT"}
EXPORTED = ("fa_fwd", "fa_fwd_kernel", "fa_bh_partition", "fa_kv_shard", "fa_fwd_kv_shard", "fa_fwd_slab", "fa_fwd_host", "fa_fwd_mma", "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_bytes", "fa_combine",
            "fa_fwd_splitkv_noalloc", "fa_fwd_fp8", "fa_fwd_blocksparse", "fa_bwd", "fa_bwd_workspace_bytes", "fa_get_device_status",
            "fa_status_string", "fa_version")


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)}")


def lib():
    """Load libfa.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "exact_attention_32_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64 = ctypes.c_void_p, ctypes.c_int64
            L.fa_fwd.restype = ctypes.c_int
            L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float,
                                 ctypes.c_int, vp]
            L.fa_fwd_kernel.restype = ctypes.c_int
            L.fa_fwd_kernel.argtypes = [i64, i64, i64, i64, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            L.fa_bh_partition.restype = ctypes.c_int
            L.fa_bh_partition.argtypes = [i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
            L.fa_kv_shard.restype = ctypes.c_int
            L.fa_kv_shard.argtypes = [i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
            L.fa_fwd_kv_shard.restype = ctypes.c_int
            L.fa_fwd_kv_shard.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                          i64, i64, vp]
            L.fa_fwd_slab.restype = ctypes.c_int
            L.fa_fwd_slab.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                      i64, i64, vp]
            L.fa_fwd_host.restype = ctypes.c_int
            L.fa_fwd_host.argtypes = [vp] * 10 + [i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, i64, vp]
            L.fa_fwd_mma.restype = ctypes.c_int
            L.fa_fwd_mma.argtypes = L.fa_fwd.argtypes
            L.fa_fwd_splitkv.restype = ctypes.c_int
            L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float,
                                         ctypes.c_int, i64, vp, i64, vp]
            L.fa_fwd_splitkv_workspace_bytes.restype = i64
            L.fa_fwd_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, i64]
            L.fa_fwd_splitkv_noalloc.restype = ctypes.c_int
            L.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float,
                                                 ctypes.c_int, i64, vp]
            L.fa_fwd_blocksparse.restype = ctypes.c_int
            L.fa_fwd_blocksparse.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float,
                                             ctypes.c_int, vp, vp]
            L.fa_fwd_fp8.restype = ctypes.c_int
            L.fa_fwd_fp8.argtypes = [vp] * 8 + [i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp]
            L.fa_bwd.restype = ctypes.c_int
            L.fa_bwd.argtypes = [vp] * 9 + [i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, vp, i64, vp]
            L.fa_bwd_workspace_bytes.restype = i64
            L.fa_bwd_workspace_bytes.argtypes = [i64] * 4
            L.fa_combine.restype = ctypes.c_int
            L.fa_combine.argtypes = [vp, vp, i64, vp, vp, i64, i64, i64, i64, vp]
            L.fa_get_device_status.restype = ctypes.c_int
            L.fa_get_device_status.argtypes = [vp]
            L.fa_status_string.restype = ctypes.c_char_p
            L.fa_status_string.argtypes = [ctypes.c_int]
            L.fa_version.restype = ctypes.c_int
            L.fa_version.argtypes = []
            _lib = L
    return _lib


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    """Raw call: pointers as ints, ``stream`` a cudaStream_t as int (0 = legacy default)."""
    return lib().fa_fwd(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), int(causal), stream)


FWD_KERNEL_NAMES = {0: "fa_fwd_tc_kernel", 1: "fa_fwd_dp_kernel"}


def fa_fwd_kernel(B: int, H: int, N: int, d: int, causal: bool) -> str:
    """Name of the kernel fa_fwd launches for these sizes (pure host
    computation in the library).  Raises FAError on invalid sizes."""
    kid = ctypes.c_int(-1)
    st = lib().fa_fwd_kernel(int(B), int(H), int(N), int(d), int(bool(causal)), ctypes.byref(kid))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_kernel")
    return FWD_KERNEL_NAMES[kid.value]


def fa_bh_partition(n_slices: int, world: int, rank: int):
    """(begin, count): the contiguous slab of (b, h) slices rank ``rank`` of
    ``world`` takes (pure host computation in the library).  Raises FAError
    on invalid arguments."""
    begin, count = ctypes.c_int64(0), ctypes.c_int64(0)
    st = lib().fa_bh_partition(int(n_slices), int(world), int(rank), ctypes.byref(begin), ctypes.byref(count))
    if st != FA_OK:
        raise FAError(st, "fa_bh_partition")
    return begin.value, count.value


def fa_kv_shard(N: int, world: int, rank: int):
    """(begin, count): the keys of every (b, h) slice that rank ``rank`` of
    ``world`` holds in a sequence-sharded problem (pure host computation in the
    library).  Raises FAError on invalid arguments."""
    begin, count = ctypes.c_int64(0), ctypes.c_int64(0)
    st = lib().fa_kv_shard(int(N), int(world), int(rank), ctypes.byref(begin), ctypes.byref(count))
    if st != FA_OK:
        raise FAError(st, "fa_kv_shard")
    return begin.value, count.value


def fa_fwd_kv_shard(q, k_shard, v_shard, o_part, lse_part, B, H, N, d, scale, causal, rank, world, stream) -> int:
    """Raw call of one rank's partial forward over its key shard."""
    return lib().fa_fwd_kv_shard(q, k_shard, v_shard, o_part, lse_part, B, H, N, d, scale, int(causal), rank,
                                 world, stream)


def fa_fwd_slab(q, k, v, o, lse, B, H, N, d, scale, causal, rank, world, stream) -> int:
    """Raw call of the forward over one rank's slab of a [B, H, N, d] problem."""
    return lib().fa_fwd_slab(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), int(causal), rank, world, stream)


def fa_fwd_host(q, k, v, o, lse, q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, N, d, scale, causal, n_groups,
                stream) -> int:
    """Raw call of the forward on host buffers (q..lse host, *_dev device staging)."""
    return lib().fa_fwd_host(q, k, v, o, lse, q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, N, d,
                             ctypes.c_float(scale), int(causal), n_groups, stream)


def fa_fwd_mma(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    """Raw call of the warp-level (mma.sync) kernel; same contract as ``fa_fwd``."""
    return lib().fa_fwd_mma(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), int(causal), stream)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, n_splits, workspace,
                   workspace_bytes, stream) -> int:
    """Raw call of the split-KV forward (caller-owned workspace)."""
    return lib().fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), int(causal),
                                n_splits, workspace, workspace_bytes, stream)


def fa_fwd_splitkv_workspace_bytes(B, H, N, d, n_splits) -> int:
    return lib().fa_fwd_splitkv_workspace_bytes(B, H, N, d, n_splits)


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, N, d, scale, causal, n_splits, stream) -> int:
    """Raw call of the split-KV forward whose scratch is the library's static
    device array: for callers that cannot allocate device memory."""
    return lib().fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), int(causal),
                                        n_splits, stream)


def fa_fwd_blocksparse(q, k, v, o, lse, B, H, N, d, scale, causal, block_mask, stream) -> int:
    """Raw call of the block-sparse forward (uint8 [nb][nb] device mask)."""
    return lib().fa_fwd_blocksparse(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), int(causal),
                                    block_mask, stream)


def fa_fwd_fp8(q, k, v, qs, ks, vs, o, lse, B, H, N, d, scale, causal, stream) -> int:
    """Raw call of the E4M3 forward (per-(b, h) fp32 scales)."""
    return lib().fa_fwd_fp8(q, k, v, qs, ks, vs, o, lse, B, H, N, d, ctypes.c_float(scale), int(causal), stream)


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes,
           stream) -> int:
    """Raw call of the backward (caller-owned workspace)."""
    return lib().fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, ctypes.c_float(scale), int(causal),
                        workspace, workspace_bytes, stream)


def fa_bwd_workspace_bytes(B, H, N, d) -> int:
    return lib().fa_bwd_workspace_bytes(B, H, N, d)


def fa_combine(o_parts, lse_parts, n_parts, o, lse, B, H, N, d, stream) -> int:
    """Raw call of the merge of partial (O, LSE) results."""
    return lib().fa_combine(o_parts, lse_parts, n_parts, o, lse, B, H, N, d, stream)


def fa_get_device_status(stream=0) -> int:
    return lib().fa_get_device_status(stream)


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def fa_version() -> int:
    return lib().fa_version()


def default_scale(d: int) -> float:
    """fp32 value of 1/sqrt(d) as a Python float."""
    return float(np.float32(1.0 / math.sqrt(d)))


def forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
            causal: bool = False, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
            stream: torch.cuda.Stream | None = None, kernel: str = "tc"):
    """O, LSE = attention(q, k, v) on the GPU through ``fa_fwd``.

    q, k, v: bf16 CUDA tensors [B, H, N, d], contiguous.  Returns (O bf16
    [B, H, N, d], LSE fp32 [B, H, N]); ``out``/``lse`` may be given to write
    in place.  Enqueued on ``stream`` (default: torch's current stream).
    ``kernel="mma"`` runs the warp-level ``fa_fwd_mma`` kernel instead of the
    tcgen05 ``fa_fwd`` kernel.
    """
    if kernel not in ("tc", "mma"):
        raise ValueError("kernel must be 'tc' or 'mma'")
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must all be [B, H, N, d]")
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = default_scale(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, N]")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        call = fa_fwd if kernel == "tc" else fa_fwd_mma
        st = call(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    B, H, N, d, float(scale), bool(causal), s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd" if kernel == "tc" else "fa_fwd_mma")
    return out, lse


def host_staging(shape, device):
    """Device staging buffers for ``forward_host``: (q, k, v, o) bf16 and lse fp32."""
    B, H, N, d = shape
    t = [torch.empty(shape, dtype=torch.bfloat16, device=device) for _ in range(4)]
    return (*t, torch.empty((B, H, N), dtype=torch.float32, device=device))


def forward_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
                 causal: bool = False, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 staging=None, n_groups: int = 0, device=None, stream: torch.cuda.Stream | None = None):
    """O, LSE = attention(q, k, v) for HOST (CPU) tensors through ``fa_fwd_host``:
    copies in, forward and copies out pipelined over groups of (b, h) slices.

    q, k, v: contiguous bf16 CPU tensors [B, H, N, d] (pinned for full copy
    speed).  ``staging`` is the tuple of device buffers from ``host_staging``
    (allocated on ``device``, default the current CUDA device, when not given).
    Returns host (O, LSE); the call is asynchronous on ``stream``: synchronise
    it before reading them.
    """
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must all be [B, H, N, d]")
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CPU tensors")
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if staging is None:
        staging = host_staging(q.shape, dev)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 CPU tensor shaped like q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CPU tensor [B, H, N]")
    qd, kd, vd, od, ld = staging
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), ld.data_ptr(),
                         B, H, N, d, float(scale), bool(causal), int(n_groups), s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_host")
    return out, lse


def forward_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_splits: int,
                    scale: float | None = None, causal: bool = False,
                    workspace: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None):
    """O, LSE by ``fa_fwd_splitkv``; the workspace (uint8 CUDA tensor) is
    allocated with torch when not given.  Returns (O, LSE, workspace)."""
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors of one shape")
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    need = fa_fwd_splitkv_workspace_bytes(B, H, N, d, n_splits)
    if need < 0:
        raise FAError(1, "fa_fwd_splitkv_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, N, d, float(scale), bool(causal), n_splits, workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_splitkv")
    return o, lse, workspace


def combine(o_parts: torch.Tensor, lse_parts: torch.Tensor, stream: torch.cuda.Stream | None = None):
    """Merge partial results: o_parts fp32 [S, B, H, N, d], lse_parts fp32
    [S, B, H, N] -> (O bf16 [B, H, N, d], LSE fp32 [B, H, N]) by ``fa_combine``."""
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32 or o_parts.dim() != 5:
        raise ValueError("o_parts must be fp32 [S, B, H, N, d] and lse_parts fp32 [S, B, H, N]")
    if not (o_parts.is_cuda and lse_parts.is_cuda and o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("o_parts and lse_parts must be contiguous CUDA tensors")
    S, B, H, N, d = o_parts.shape
    if tuple(lse_parts.shape) != (S, B, H, N):
        raise ValueError("lse_parts must be [S, B, H, N]")
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=o_parts.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=o_parts.device)
    s = stream if stream is not None else torch.cuda.current_stream(o_parts.device)
    with torch.cuda.device(o_parts.device):
        st = fa_combine(o_parts.data_ptr(), lse_parts.data_ptr(), S, o.data_ptr(), lse.data_ptr(),
                        B, H, N, d, s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_combine")
    return o, lse


def forward_kv_shard(q: torch.Tensor, k_shard: torch.Tensor | None, v_shard: torch.Tensor | None, rank: int,
                     world: int, scale: float | None = None, causal: bool = False,
                     stream: torch.cuda.Stream | None = None):
    """This rank's partial (O fp32 [B, H, N, d], LSE fp32 [B, H, N]) of a
    sequence-sharded forward by ``fa_fwd_kv_shard``: all query rows of q
    against the keys ``fa_kv_shard(N, world, rank)`` gives, held in k_shard and
    v_shard ([B, H, count, d] bf16 CUDA tensors; None when count is 0)."""
    if q.dim() != 4 or q.dtype != torch.bfloat16 or not q.is_cuda or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 CUDA tensor [B, H, N, d]")
    B, H, N, d = q.shape
    begin, count = fa_kv_shard(N, world, rank)
    if count > 0:
        for t in (k_shard, v_shard):
            if (t is None or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous()
                    or tuple(t.shape) != (B, H, count, d)):
                raise ValueError(f"k_shard and v_shard must be contiguous bf16 CUDA tensors [{B}, {H}, {count}, {d}]")
    scale = default_scale(d) if scale is None else scale
    o_part = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    lse_part = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    kp = k_shard.data_ptr() if count > 0 else None
    vp = v_shard.data_ptr() if count > 0 else None
    with torch.cuda.device(q.device):
        st = fa_fwd_kv_shard(q.data_ptr(), kp, vp, o_part.data_ptr(), lse_part.data_ptr(), B, H, N, d, scale,
                             causal, rank, world, s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_kv_shard")
    return o_part, lse_part


def gather_parts(o_part: torch.Tensor, lse_part: torch.Tensor, group=None):
    """The exchange step of a sequence-sharded forward: all-gather every rank's
    partial (O, LSE) over ``torch.distributed`` into ([world, ...], [world, ...])
    tensors, in rank order, ready for ``combine``."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    o_list = [torch.empty_like(o_part) for _ in range(world)]
    lse_list = [torch.empty_like(lse_part) for _ in range(world)]
    dist.all_gather(o_list, o_part.contiguous(), group=group)
    dist.all_gather(lse_list, lse_part.contiguous(), group=group)
    return torch.stack(o_list), torch.stack(lse_list)


def forward_sequence_sharded(q: torch.Tensor, k_shard: torch.Tensor | None, v_shard: torch.Tensor | None,
                             scale: float | None = None, causal: bool = False, group=None):
    """(O bf16, LSE) of the whole problem on every rank of ``group``: this
    rank's partial (``forward_kv_shard``), the all-gather of the parts
    (``gather_parts``), and their merge (``combine``)."""
    import torch.distributed as dist
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    o_part, lse_part = forward_kv_shard(q, k_shard, v_shard, rank, world, scale=scale, causal=causal)
    o_parts, lse_parts = gather_parts(o_part, lse_part, group)
    return combine(o_parts, lse_parts)


def backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
             dout: torch.Tensor, scale: float | None = None, causal: bool = False,
             workspace: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None):
    """(dQ, dK, dV) by ``fa_bwd``; o and lse are ``forward``'s outputs.  The
    workspace (uint8 CUDA tensor) is allocated with torch when not given."""
    for t in (q, k, v, o, dout):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError("q, k, v, o, dout must be contiguous bf16 CUDA tensors of one shape")
    B, H, N, d = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, H, N]")
    scale = default_scale(d) if scale is None else scale
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if need < 0:
        raise FAError(1 if d in (64, 128) else 2, "fa_bwd_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                    dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, float(scale), bool(causal),
                    workspace.data_ptr(), workspace.numel() * workspace.element_size(), s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_bwd")
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    """fa_fwd in the forward, fa_bwd in the backward (O and LSE saved)."""

    @staticmethod
    def forward(ctx, q, k, v, scale, causal):
        o, lse = forward(q, k, v, scale=scale, causal=causal)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale, ctx.causal = scale, causal
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = backward(q, k, v, o, lse, dout.contiguous(), scale=ctx.scale, causal=ctx.causal)
        return dq, dk, dv, None, None


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
              causal: bool = False) -> torch.Tensor:
    """O = attention(q, k, v) with autograd: ``fa_fwd`` forward, ``fa_bwd``
    backward (dQ, dK, dV of the loss through O).  q, k, v: contiguous bf16
    CUDA tensors [B, H, N, d] (d = 64 or 128)."""
    return _Attention.apply(q, k, v, default_scale(q.shape[-1]) if scale is None else scale, bool(causal))


def forward_fp8(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, q_scale: torch.Tensor,
                k_scale: torch.Tensor, v_scale: torch.Tensor, scale: float | None = None,
                causal: bool = False, stream: torch.cuda.Stream | None = None):
    """(O bf16, LSE fp32) by ``fa_fwd_fp8``: q8, k8, v8 are float8_e4m3fn (or
    uint8) CUDA tensors [B, H, N, 128]; the scales fp32 [B, H] (or [B*H])."""
    for t in (q8, k8, v8):
        if t.element_size() != 1 or not t.is_cuda or not t.is_contiguous() or t.shape != q8.shape:
            raise ValueError("q8, k8, v8 must be contiguous 8-bit CUDA tensors of one shape")
    B, H, N, d = q8.shape
    for t in (q_scale, k_scale, v_scale):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.numel() != B * H:
            raise ValueError("scales must be contiguous fp32 CUDA tensors with B*H elements")
    scale = default_scale(d) if scale is None else scale
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    s = stream if stream is not None else torch.cuda.current_stream(q8.device)
    with torch.cuda.device(q8.device):
        st = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), q_scale.data_ptr(), k_scale.data_ptr(),
                        v_scale.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, float(scale),
                        bool(causal), s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    return o, lse


def forward_blocksparse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_mask: torch.Tensor,
                        scale: float | None = None, causal: bool = False,
                        stream: torch.cuda.Stream | None = None):
    """(O, LSE) by ``fa_fwd_blocksparse``; block_mask is a 0/1 tensor
    [ceil(N/128), ceil(N/128)] (moved to the device as uint8)."""
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors of one shape")
    B, H, N, d = q.shape
    nb = -(-N // 128)
    if tuple(block_mask.shape) != (nb, nb):
        raise ValueError(f"block_mask must be [{nb}, {nb}]")
    bm = (block_mask != 0).to(device=q.device, dtype=torch.uint8).contiguous()
    scale = default_scale(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa_fwd_blocksparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, H, N, d, float(scale), bool(causal), bm.data_ptr(), s.cuda_stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_blocksparse")
    return o, lse
