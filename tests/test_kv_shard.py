"""Sequence sharding: every rank holds all queries and one contiguous range of
the keys, computes its partial (O, LSE), and the parts are gathered and merged
with the two-block merge ("FlashAttention: IO-Aware Tiling, Online Softmax
Mathematics, ...", section "Online Softmax Mathematics").

CPU: the key partition (fa_kv_shard) and its argument checks; the exchange
(gather_parts over gloo, world 2 and 3) on parts the oracle computes, merged by
the oracle, against the oracle's whole result.
GPU: the ranks run one after another on one GPU (fa_fwd_kv_shard on each
rank's own K and V rows); every part against the oracle restricted to that
key range, the merged parts against the oracle, and bit for bit against
fa_fwd_splitkv with n_splits = world (the same ranges).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import exact_attention_32_gb300 as fa
from exact_attention_32_gb300 import make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MAX_O, MEAN_O, MAX_LSE = 2e-2, 2e-3, 1e-3


def test_partition_covers_every_key_once_in_128_key_ranges():
    for N in list(range(1, 300)) + [1000, 4096, 16384, 16385, 131072]:
        for world in (1, 2, 3, 4, 5, 7, 8, 16, 32):
            shards = [fa.fa_kv_shard(N, world, r) for r in range(world)]
            per = -(-N // world)
            chunk = -(-per // 128) * 128
            pos = 0
            for r, (begin, count) in enumerate(shards):
                assert begin == min(r * chunk, N)                # split r of fa_fwd_splitkv
                assert begin == pos and 0 <= count <= chunk      # contiguous, in rank order
                assert begin % 128 == 0 or count == 0
                pos += count
            assert pos == N


@pytest.mark.parametrize("args", [(0, 2, 0), (100, 0, 0), (100, 33, 0), (100, 2, 2), (100, 2, -1)])
def test_partition_rejects_bad_arguments(args):
    with pytest.raises(fa.FAError):
        fa.fa_kv_shard(*args)


def test_shard_forward_rejects_bad_arguments_before_any_device_call():
    L = fa.lib()
    # bad rank / world, bad sizes, bad scale: refused on the host
    for rank, world, N, scale in [(2, 2, 256, 0.125), (0, 0, 256, 0.125), (0, 33, 256, 0.125),
                                  (0, 2, 0, 0.125), (0, 2, 256, 0.0)]:
        assert L.fa_fwd_kv_shard(16, 16, 16, 16, 16, 1, 1, N, 64, scale, 0, rank, world, None) == 1


def oracle_part(q, k, v, scale, causal, begin, count):
    """The oracle over keys [begin, begin + count); a rank with no key has no
    admitted key in any row: O = 0, LSE = -inf."""
    if count == 0:
        B, H, N, d = q.shape
        return np.zeros((B, H, N, d)), np.full((B, H, N), -np.inf)
    return oracle.attention(q, k, v, scale, causal, kv_range=(begin, begin + count))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _exchange_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import exact_attention_32_gb300 as fa
    from exact_attention_32_gb300 import make_inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    for N, causal in [(300, True), (200, False), (1000, True)]:
        q, k, v = make_inputs(1, 2, N, 64, seed=40 + N)
        begin, count = fa.fa_kv_shard(N, world, rank)
        o_part, lse_part = oracle_part(q, k, v, 0.125, causal, begin, count)
        o_parts, lse_parts = fa.gather_parts(torch.from_numpy(o_part), torch.from_numpy(lse_part))
        out[(rank, N)] = (o_parts.numpy(), lse_parts.numpy())
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_over_gloo_gives_the_whole_result(world):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_exchange_worker, args=(world, free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for N, causal in [(300, True), (200, False), (1000, True)]:
        q, k, v = make_inputs(1, 2, N, 64, seed=40 + N)
        o_ref, lse_ref = oracle.attention(q, k, v, 0.125, causal)
        o_parts, lse_parts = out[(0, N)]
        for r in range(1, world):  # every rank received the same parts, in rank order
            assert np.array_equal(out[(r, N)][0], o_parts) and np.array_equal(out[(r, N)][1], lse_parts)
        for r in range(world):
            begin, count = fa.fa_kv_shard(N, world, r)
            o_r, lse_r = oracle_part(q, k, v, 0.125, causal, begin, count)
            assert np.array_equal(o_parts[r], o_r) and np.array_equal(lse_parts[r], lse_r)
        o_m, lse_m = oracle.merge(o_parts, lse_parts)
        assert np.abs(o_m - o_ref).max() < 1e-12 and np.abs(lse_m - lse_ref).max() < 1e-12


def run_ranks(q, k, v, world, scale, causal):
    """Every rank's fa_fwd_kv_shard, one after another on this GPU, each given
    only its own rows of K and V."""
    N = q.shape[2]
    parts = []
    for r in range(world):
        begin, count = fa.fa_kv_shard(N, world, r)
        ks = k[:, :, begin:begin + count].contiguous().cuda() if count else None
        vs = v[:, :, begin:begin + count].contiguous().cuda() if count else None
        parts.append(fa.forward_kv_shard(q.cuda(), ks, vs, r, world, scale=scale, causal=causal))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(0) == 0
    return torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts])


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,world", [(1, 2), (200, 3), (300, 2), (1000, 3), (1000, 8), (640, 5), (4096, 4)])
def test_shards_merge_to_the_whole_result(N, world, d, causal):
    q, k, v = make_inputs(2, 2, N, d, seed=700 + N + world + d + causal)
    scale = float(np.float32(1 / np.sqrt(d)))
    o_parts, lse_parts = run_ranks(q, k, v, world, scale, causal)
    # each part: the attention over its key range alone
    for r in range(world):
        begin, count = fa.fa_kv_shard(N, world, r)
        op_ref, lp_ref = oracle_part(q, k, v, scale, causal, begin, count)
        op, lp = o_parts[r].double().cpu().numpy(), lse_parts[r].double().cpu().numpy()
        empty = np.isneginf(lp_ref)
        assert np.array_equal(np.isneginf(lp), empty)
        assert np.all(op[empty] == 0.0)
        if (~empty).any():
            err = np.abs(op[~empty] - op_ref[~empty])
            assert err.max() <= MAX_O and err.mean() <= MEAN_O
            assert np.abs(lp[~empty] - lp_ref[~empty]).max() <= MAX_LSE
    # merged: the whole problem, and exactly what the one-GPU split-KV forward gives
    o, lse = fa.combine(o_parts, lse_parts)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    err = np.abs(o.double().cpu().numpy() - o_ref)
    assert err.max() <= MAX_O and err.mean() <= MEAN_O
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= MAX_LSE
    o_s, lse_s, _ = fa.forward_splitkv(q.cuda(), k.cuda(), v.cuda(), world, scale=scale, causal=causal)
    chunk = -(-(-(-N // world)) // 128) * 128
    parts = -(-N // chunk)  # key ranges fa_fwd_splitkv merges (ranks past them hold no key)
    if parts == world:  # with empty shards the merge folds extra empty parts: equal up to rounding
        assert torch.equal(o, o_s) and torch.equal(lse, lse_s)
    else:
        assert (o.float() - o_s.float()).abs().max().item() <= 2 ** -7


def _nccl_one_rank_worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import exact_attention_32_gb300 as fa
    from exact_attention_32_gb300 import make_inputs
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    q, k, v = make_inputs(2, 3, 700, 128, seed=77)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.forward_sequence_sharded(qc, kc, vc, scale=0.08838834764831845, causal=True)
    o_s, lse_s, _ = fa.forward_splitkv(qc, kc, vc, 1, scale=0.08838834764831845, causal=True)
    torch.cuda.synchronize()
    out["equal"] = bool(torch.equal(o, o_s) and torch.equal(lse, lse_s))
    out["status"] = fa.fa_get_device_status(0)
    dist.destroy_process_group()


@pytest.mark.gpu
def test_sequence_sharded_forward_through_nccl_on_one_rank():
    # the product function end to end: the shard forward, the NCCL all-gather
    # (one rank) and the merge give the split-KV forward's result bit for bit
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_nccl_one_rank_worker, args=(free_port(), out), nprocs=1, join=True, start_method="spawn")
    assert out["status"] == 0 and out["equal"]
