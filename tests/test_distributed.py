"""The multi-process path on CPU: gloo, world sizes 2 and 3.

Attention over (b, h) slices has no exchange step ("6.1 FlashAttention V1 in
detail", section 8.2), so a job is sharded by giving each rank a contiguous
slab of slices (the library's fa_bh_partition) and each rank runs the forward
on its slab alone.  The tests check that the slabs cover every slice exactly
once for uneven slice counts, that the slab inputs the bench gives each rank,
run through the oracle and gathered, are the whole job's result, and that the
only collectives (barrier, max-reduce of timings) work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup(None)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(float(10 * rank + 1), w)
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(2, free_port(), out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 11.0, 1: 11.0}


def _slab_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    import exact_attention_32_gb300 as fa
    bench.dist_setup(None)
    # every slice count from 0 to 3 * world + 2: gather the slabs of all ranks
    slabs = {}
    for n in range(3 * world + 3):
        mine = fa.fa_bh_partition(n, world, rank)
        got = [None] * world
        dist.all_gather_object(got, mine)
        slabs[n] = got
    out[("slabs", rank)] = slabs
    # the bench's slab inputs on a small workload, through the oracle
    import oracle
    from exact_attention_32_gb300.workloads import Workload
    w = Workload("tiny", 1, 5, 64, 64, True, 1.0, 3)
    for scaling in ("weak", "strong"):
        shape, (q, k, v), flops, (begin, count) = bench.slab_inputs(w, world, rank, scaling)
        o, lse = oracle.attention(q, k, v, w.scale, w.causal) if count else (None, None)
        got = [None] * world
        dist.all_gather_object(got, (begin, count, None if o is None else o.reshape(-1, 64), flops))
        out[(scaling, rank)] = got
    dist.destroy_process_group()


def run_slab_workers(world):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_slab_worker, args=(world, free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    return dict(out)


@pytest.mark.parametrize("world", [2, 3])
def test_slabs_cover_every_slice_once_and_give_the_whole_result(world):
    import numpy as np
    import oracle
    from exact_attention_32_gb300 import workload_inputs
    from exact_attention_32_gb300.workloads import Workload
    out = run_slab_workers(world)
    for rank in range(world):
        assert out[("slabs", rank)] == out[("slabs", 0)]  # every rank sees the same partition
    for n, slabs in out[("slabs", 0)].items():
        owner = np.zeros(n, dtype=int)
        for begin, count in slabs:
            owner[begin:begin + count] += 1
        assert (owner == 1).all(), (n, slabs)                        # each slice exactly once
        assert [b for b, _ in slabs] == sorted(b for b, _ in slabs)  # contiguous, in rank order
        counts = [c for _, c in slabs]
        assert max(counts) - min(counts) <= 1                        # balanced
    w = Workload("tiny", 1, 5, 64, 64, True, 1.0, 3)
    # strong: the ranks' results, gathered in slab order, are the workload's result
    got = out[("strong", 0)]
    o_ref, _ = oracle.attention(*workload_inputs(w), w.scale, w.causal)
    parts = [o for _, c, o, _ in got if c]
    assert np.array_equal(np.concatenate(parts), o_ref.reshape(-1, 64))
    assert all(f == w.flops for *_, f in got)
    # weak: rank r's slab is draw r of the workload (seed + r), the job world draws
    got = out[("weak", 0)]
    for r, (begin, count, o, flops) in enumerate(got):
        assert (begin, count) == (r * 5, 5) and flops == world * w.flops
        o_r, _ = oracle.attention(*workload_inputs(w, seed=w.seed + r), w.scale, w.causal)
        assert np.array_equal(o, o_r.reshape(-1, 64))


def test_partition_rejects_bad_arguments():
    import exact_attention_32_gb300 as fa
    for args in [(-1, 2, 0), (4, 0, 0), (4, 2, 2), (4, 2, -1)]:
        with pytest.raises(fa.FAError):
            fa.fa_bh_partition(*args)
    assert fa.fa_bh_partition(0, 3, 2) == (0, 0)


def test_bench_reference_arm_under_torchrun():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "b1_h1_n256_d64"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["workload"] == "b1_h1_n256_d64"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
