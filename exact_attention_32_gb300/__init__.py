"""GB300-native exact attention forward (sm_103a).

``forward(q, k, v, scale=None, causal=False)`` returns (O, LSE) computed by the
CUDA kernels of ``libfa.so`` (see include/fa.h); the raw C ABI is exposed under
its own names (``fa_fwd``, ``fa_fwd_host``, ``fa_fwd_mma``, ``fa_get_device_status``,
``fa_status_string``, ``fa_version``, ...).  ``forward_host`` runs the forward on
host tensors with the copies overlapped.  The library is loaded on first use and its absence raises.
"""
from ._binding import (FAError, attention, backward, combine, default_scale, fa_bwd, fa_bwd_workspace_bytes,  # noqa: F401
                       fa_bh_partition, fa_kv_shard, fa_fwd_kv_shard, forward_kv_shard, gather_parts,
                       forward_sequence_sharded, fa_combine, fa_fwd_slab, fa_fwd, fa_fwd_kernel, fa_fwd_blocksparse, fa_fwd_fp8, fa_fwd_host, fa_fwd_mma,
                       forward_blocksparse, forward_fp8, forward_host, host_staging,
                       fa_fwd_splitkv, fa_fwd_splitkv_noalloc, fa_fwd_splitkv_workspace_bytes,
                       fa_get_device_status,
                       fa_status_string, fa_version, forward, forward_splitkv, lib)
from .workloads import HEADLINE, WORKLOADS, Workload, make_inputs, workload_inputs  # noqa: F401
