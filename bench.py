#!/usr/bin/env python
"""Benchmark: fused exact attention forward on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one forward pass (one fa_fwd launch) over the whole workload, with
inputs resident in device memory.  The default workload is the long causal
run B=1, H=32, N=16384, d=128.  Q/K/V (402 MB) plus O (134 MB) exceed the
129 MB L2, so consecutive steps do not run from a warm L2.

Under torchrun (N > 1) the job is sharded over the ranks by (b, h) slices:
rank r takes the contiguous slab fa_bh_partition(B*H, N, r) and runs fa_fwd
on it on its own GPU.  The slices are independent, so no collective touches
the data (a barrier and a max-reduce of the timings only).  ``--scaling
weak`` (default): the job is N draws of the workload (draw r from seed
seed + r, draw 0 the workload itself), B*H*N slices in all, so every rank
keeps the workload's size.  ``--scaling strong``: the job is the workload
itself, its B*H slices split over the ranks.

``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample of
rows of the same workload, and reports the same metric for it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_attention_32_gb300.workloads import HEADLINE, WORKLOADS, workload_inputs  # noqa: E402

L2_BYTES = 129 * 1000 * 1000  # GB300 L2 (129 MB)
METRIC = "attention fwd TFLOPS (bf16, 1×GB300) and % of dense BF16 tensor peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
KERNEL_SOURCES = {"fa_fwd_tc_kernel": "exact_attention_32_gb300/csrc/fa_fwd_tc.cu",
                  "fa_fwd_dp_kernel": "exact_attention_32_gb300/csrc/fa_fwd_dp.cu",
                  "fa_fwd_mma_kernel": "exact_attention_32_gb300/csrc/fa_fwd_mma.cu"}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--kernel", default="tc", choices=["tc", "mma"],
                   help="forward kernel of the timed step: tc = fa_fwd (tcgen05, the product path), "
                        "mma = fa_fwd_mma (the warp-level mma.sync kernel, kept as a baseline)")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--scaling", default="weak", choices=["weak", "strong"],
                   help="under torchrun: weak = N draws of the workload, one slab of B*H slices per rank; "
                        "strong = the workload's B*H slices split over the ranks")
    p.add_argument("--shard", default="heads", choices=["heads", "seq"],
                   help="under torchrun: heads = slabs of (b, h) slices, no exchange (the default); seq = every "
                        "rank holds all queries and one key shard (fa_fwd_kv_shard), then an all-gather of the "
                        "partial (O, LSE) and their merge (fa_combine); strong scaling over the workload's keys")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-secondary", action="store_true",
                   help="skip the secondary rows: split-KV merge, backward, FP8 and block-sparse forward")
    return p.parse_args()


# ----------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def slab_inputs(w, world: int, rank: int, scaling: str):
    """This rank's part of the job: (local shape (B, H, N, d), CPU inputs
    (q, k, v) of that shape, FLOPs of the whole job, slab (begin, count) in
    the job's (b, h) slices).  The slab comes from the library's
    fa_bh_partition."""
    import exact_attention_32_gb300 as fa
    BH = w.B * w.H
    if scaling == "weak":
        # the job: `world` draws of the workload stacked along the batch (draw r
        # from seed + r); rank r's slab is exactly draw r
        begin, count = fa.fa_bh_partition(world * BH, world, rank)
        assert begin == rank * BH and count == BH
        inputs = workload_inputs(w, seed=w.seed + rank)
        return (w.B, w.H, w.N, w.d), inputs, w.flops * world, (begin, count)
    begin, count = fa.fa_bh_partition(BH, world, rank)
    q, k, v = (t.reshape(1, BH, w.N, w.d)[:, begin:begin + count].contiguous() for t in workload_inputs(w))
    return (1, count, w.N, w.d), (q, k, v), w.flops, (begin, count)


# ---------------------------------------------------------------------- peaks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch from the committed ncu summary of this
    kernel and workload, or None when absent or taken on a different source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = os.path.join(ROOT, KERNEL_SOURCES[kernel])
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_s = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m_t or not m_s or m_s.group(1) != sha:
        return None
    return float(m_t.group(1))


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 100 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.file = None
        self.target = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            self.target = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else None
        except Exception:
            self.target = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.target:
                cmd += ["-i", self.target]
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [line.strip().split(",") for line in self.file if line.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ secondary row

def combine_roofline(w, dev, peaks, peak_src, n_parts=4, steps=20):
    """fa_combine (the split-KV merge) on synthetic fp32 parts shaped like the
    workload: a memory-bound kernel, reported against the measured copy
    bandwidth.  Algorithmic bytes per launch: every part read once
    (S * rows * (4d + 4)), O and LSE written once (rows * (2d + 4))."""
    import exact_attention_32_gb300 as fa
    rows = w.B * w.H * w.N
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    o_parts = torch.randn((n_parts, w.B, w.H, w.N, w.d), generator=g).to(dev)
    lse_parts = (torch.randn((n_parts, w.B, w.H, w.N), generator=g) * 4).to(dev)
    o = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    args = (o_parts.data_ptr(), lse_parts.data_ptr(), n_parts, o.data_ptr(), lse.data_ptr(),
            w.B, w.H, w.N, w.d, stream.cuda_stream)
    for _ in range(3):
        if fa.fa_combine(*args) != 0:
            raise fa.FAError(fa.fa_combine(*args), "fa_combine")
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fa.fa_combine(*args)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    nbytes = n_parts * rows * (4 * w.d + 4) + rows * (2 * w.d + 4)
    peak = float(peaks["hbm_gbs"])
    achieved = nbytes / (ms / 1e3) / 1e9
    return {"kernel": "fa_combine_kernel", "row": "split-KV merge of partial (O, LSE)", "bound": "hbm",
            "parts": n_parts, "achieved": achieved, "peak": peak, "peak_source": f"{peak_src} hbm_gbs",
            "unit": "GB/s", "frac": achieved / peak, "algorithmic_bytes_per_launch": nbytes,
            "launch_ms": ms, "data": "synthetic fp32 parts, inputs larger than L2"}


def backward_throughput(w, dev, peaks, peak_src, steps=10):
    """fa_bwd (pre + tcgen05 main + post launches) on the workload with a seeded
    dO: conventional backward FLOPs 2.5 x the forward's (five N^2 d products
    instead of two), halved when causal."""
    import exact_attention_32_gb300 as fa
    from exact_attention_32_gb300.workloads import make_grad_output
    q, k, v = (t.to(dev) for t in workload_inputs(w))
    do = make_grad_output(w.B, w.H, w.N, w.d, w.seed, device=dev)
    o, lse = fa.forward(q, k, v, scale=w.scale, causal=w.causal)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    stream = torch.cuda.current_stream(dev)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N, w.d, w.scale, w.causal,
            ws.data_ptr(), ws.numel(), stream.cuda_stream)
    for _ in range(3):
        st = fa.fa_bwd(*args)
        if st != 0:
            raise fa.FAError(st, "fa_bwd")
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fa.fa_bwd(*args)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    flops = 2.5 * w.flops
    peak = float(peaks["bf16_tflops"])
    achieved = flops / (ms / 1e3) / 1e12
    return {"kernel": "fa_bwd_tc_kernel (+ pre, post)", "row": "backward dQ, dK, dV", "bound": "tensor",
            "achieved": achieved, "peak": peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
            "unit": "TFLOP/s", "frac": achieved / peak, "algorithmic_flops_per_step": flops,
            "ms_per_step": ms, "launches_per_step": 3}


def fp8_throughput(w, dev, peaks, peak_src, steps=20):
    """fa_fwd_fp8 on the workload encoded as E4M3 per (b, h) (power-of-two
    scales).  Peak: the measured bf16 peak times the nominal dense E4M3/bf16
    ratio of 2 (4.5 vs 2.25 PFLOP/s)."""
    import exact_attention_32_gb300 as fa
    from exact_attention_32_gb300.workloads import quantize_e4m3
    if w.d != 128:
        return None
    enc = [quantize_e4m3(t) for t in workload_inputs(w)]
    (q8, qs, _), (k8, ks, _), (v8, vs, _) = [(a.to(dev), b.to(dev), None) for a, b, _ in enc]
    o = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    args = (q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), qs.data_ptr(), ks.data_ptr(), vs.data_ptr(),
            o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N, w.d, w.scale, w.causal, stream.cuda_stream)
    for _ in range(3):
        st = fa.fa_fwd_fp8(*args)
        if st != 0:
            raise fa.FAError(st, "fa_fwd_fp8")
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fa.fa_fwd_fp8(*args)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    peak = 2.0 * float(peaks["bf16_tflops"])
    achieved = w.flops / (ms / 1e3) / 1e12
    return {"kernel": "fa_fwd_dp_kernel (E4M3)", "row": "FP8 forward", "bound": "tensor", "achieved": achieved,
            "peak": peak, "peak_source": f"{peak_src} bf16_tflops x 2 (nominal E4M3/bf16 dense ratio)",
            "unit": "TFLOP/s", "frac": achieved / peak, "algorithmic_flops_per_launch": w.flops,
            "launch_ms": ms}


def blocksparse_throughput(w, dev, peaks, peak_src, steps=20):
    """fa_fwd_blocksparse on the workload with a sliding window of three
    128-blocks plus the first block column as global keys.  Algorithmic FLOPs:
    4 d per admitted (query, key) pair (causal pairs only when causal)."""
    import exact_attention_32_gb300 as fa
    nb = -(-w.N // 128)
    i, j = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    mask = ((np.abs(i - j) <= 1) | (j == 0)).astype(np.uint8)
    # admitted pairs per slice, counted block by block (exact for causal diagonals)
    pairs = 0
    for qb in range(nb):
        qlo, qhi = qb * 128, min(w.N, qb * 128 + 128)
        for kb in np.nonzero(mask[qb])[0]:
            klo, khi = kb * 128, min(w.N, kb * 128 + 128)
            if not w.causal:
                pairs += (qhi - qlo) * (khi - klo)
            else:
                for qi in range(qlo, qhi):
                    pairs += max(0, min(khi, qi + 1) - klo)
    flops = 4.0 * w.d * pairs * w.B * w.H
    q, k, v = (t.to(dev) for t in workload_inputs(w))
    bm = torch.as_tensor(mask, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N, w.d,
            w.scale, w.causal, bm.data_ptr(), stream.cuda_stream)
    for _ in range(3):
        st = fa.fa_fwd_blocksparse(*args)
        if st != 0:
            raise fa.FAError(st, "fa_fwd_blocksparse")
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fa.fa_fwd_blocksparse(*args)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    peak = float(peaks["bf16_tflops"])
    achieved = flops / (ms / 1e3) / 1e12
    return {"kernel": "fa_fwd_tc_kernel (block-sparse)", "row": "block-sparse forward",
            "mask": "window of 3 blocks + first block column", "admitted_fraction_of_dense": flops / w.flops,
            "bound": "tensor", "achieved": achieved, "peak": peak,
            "peak_source": f"{peak_src} bf16_tflops (burst)", "unit": "TFLOP/s", "frac": achieved / peak,
            "algorithmic_flops_per_launch": flops, "launch_ms": ms}


# ------------------------------------------------------------- CPU baseline

def oracle_rows_for(w, seconds: float, threads: int, rng_seed: int = 0):
    """Evenly spaced rows of the workload whose fp64 oracle cost is about
    ``seconds`` on ``threads`` threads (calibrated on a small first batch)."""
    import oracle
    q, k, v = workload_inputs(w)
    total = w.B * w.H * w.N
    n = max(threads * 2, 8)
    while True:
        calib = np.linspace(0, total - 1, min(n, total)).round().astype(np.int64)
        t0 = time.perf_counter()
        oracle.attention(q, k, v, w.scale, w.causal, rows=calib, threads=threads)
        dt = time.perf_counter() - t0
        if dt >= min(0.5, seconds / 4) or n >= total:
            break
        n *= 4
    per_row = dt / len(calib)
    n = int(min(total, max(len(calib), seconds / max(per_row, 1e-9))))
    rows = np.unique(np.linspace(0, total - 1, n).round().astype(np.int64))
    return (q, k, v), rows


def time_oracle(w, inputs, rows, threads):
    import oracle
    q, k, v = inputs
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.causal, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    # conventional work of those rows: the workload's FLOPs spread evenly over its rows
    flops = w.flops * len(rows) / (w.B * w.H * w.N)
    return dt, flops


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, seconds):
    threads = cpu_threads()
    inputs, rows = oracle_rows_for(w, seconds, threads)
    dt, flops = time_oracle(w, inputs, rows, threads)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} evenly spaced query rows of {w.B * w.H * w.N} "
                      f"({w.name}), fp64 C oracle, {dt:.1f} s"}


# ------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import exact_attention_32_gb300 as fa

    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", local if world > 1 else 0)
    fa.lib()
    (Bl, Hl, N, d), (q_h, k_h, v_h), job_flops, slab = slab_inputs(w, world, rank, args.scaling)
    local_flops = w.flops / (w.B * w.H) * Bl * Hl  # this rank's share
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty(Bl, Hl, N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
    busy = Bl * Hl > 0  # a strong-scaling rank past the last slice has nothing to run

    fwd = fa.fa_fwd if args.kernel == "tc" else fa.fa_fwd_mma
    # fa_fwd hands d = 64 problems of short units to its second kernel; the
    # roofline names the kernel that actually runs
    if args.kernel == "mma":
        kernel_name = "fa_fwd_mma_kernel"
    else:
        kernel_name = fa.fa_fwd_kernel(Bl, Hl, N, d, w.causal) if busy else "fa_fwd_tc_kernel"

    def step():
        if not busy:
            return
        st = fwd(*ptrs, Bl, Hl, N, d, w.scale, w.causal, sp)
        if st != 0:
            raise fa.FAError(st, "fa_fwd" if args.kernel == "tc" else "fa_fwd_mma")

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # inputs smaller than L2 are evicted between steps by writing a 256 MB
    # buffer (outside the per-launch events; `value` then comes from those)
    io_bytes = 4 * Bl * Hl * N * d * 2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if busy and io_bytes < 2 * L2_BYTES else None
    # the clock sampler starts before the warm-up, so that the timed steps follow
    # the warm-up steps directly (an idle GPU runs its first launches slower)
    clocks = ClockSampler(dev.index) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    for i in range(args.warmup):
        if flush is not None:
            flush.fill_(i & 255)
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 255)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop() if clocks else None
    st = fa.fa_get_device_status(sp)
    if st != 0:
        raise fa.FAError(st, "warm-up or timed region")
    total_ms = max_over_ranks(e0.elapsed_time(e1), world)
    durations = sorted(s.elapsed_time(e) for s, e in zip(starts, ends))
    launch_ms = max_over_ranks(statistics.mean(durations), world)
    # the distribution of this rank's per-launch times (nearest-rank percentiles)
    pct = {f"p{q}": durations[min(len(durations) - 1, max(0, round(q / 100 * len(durations)) - 1))]
           for q in (10, 50, 90)}

    if flush is not None:  # the timed region also holds the flushes: count the launches only
        total_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)), world)
    value = job_flops * K / (total_ms / 1e3) / 1e12

    # end to end through the C ABI with host buffers (fa_fwd_host): pinned host
    # Q, K, V in, O and LSE out, every copy inside the timed region; the
    # library overlaps the copies of one group of (b, h) slices with the
    # forward of another
    e2e = None
    if not args.no_e2e and busy:
        qp, kp, vp_ = (t.pin_memory() for t in (q_h, k_h, v_h))
        op = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        lp = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        staging = (q, k, v, o, lse)

        def e2e_step():
            fa.forward_host(qp, kp, vp_, scale=w.scale, causal=w.causal, out=op, lse=lp, staging=staging,
                            device=dev, stream=stream)

        for _ in range(3):
            e2e_step()
        Ke = max(3, min(K, 30))
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(Ke):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
        out_bytes = o.numel() * o.element_size() + lse.numel() * lse.element_size()
        e2e = {"value": job_flops * Ke / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "steps": Ke, "ms_per_step": e2e_ms / Ke,
               "api": "fa_fwd_host (pinned host buffers, copies overlapped over 8 groups of (b, h) slices)"}

    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = local_flops / (launch_ms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": args.scaling, "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: Q, K, V iid N(0,1) fp32 rounded to bf16, seeded",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "scale": w.scale,
                   "global_batch": w.B * world if args.scaling == "weak" else w.B,
                   "seq_len": w.N, "parallelism": f"bh_slabs{world}",
                   "slab_rank0": {"begin": slab[0], "count": slab[1]},
                   "l2": ("inputs larger than L2 (Q+K+V+O exceed 2 x 129 MB), no flush" if flush is None else
                          "L2 flushed between steps (256 MB write, outside the per-launch events); "
                          "value from the per-launch event times")},
        "pct_of_dense_bf16_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "kernel": kernel_name, "achieved": achieved,
                     "peak": peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": load_traffic(kernel_name, w.name) if Bl * Hl == w.B * w.H else None,
                     "algorithmic_flops_per_launch": local_flops,
                     "algorithmic_bytes_per_launch": w.min_bytes // (w.B * w.H) * Bl * Hl,
                     "launch_ms": launch_ms},
        "gpu_launches": K,
        "launch_ms_percentiles": pct,
        "max_memory_allocated_bytes": torch.cuda.max_memory_allocated(dev),
        "impl": "ours",
    }
    if e2e:
        line["e2e"] = e2e
    line["clocks"] = clk
    if not args.no_secondary:
        sec = [combine_roofline(w, dev, peaks, peak_src), backward_throughput(w, dev, peaks, peak_src),
               fp8_throughput(w, dev, peaks, peak_src), blocksparse_throughput(w, dev, peaks, peak_src)]
        line["secondary"] = [x for x in sec if x is not None]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return line


# ------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    threads = cpu_threads()
    budget = 150.0  # seconds of oracle work for the whole run
    per_step = budget / max(1, args.steps + args.warmup)
    inputs, rows = oracle_rows_for(w, per_step, threads)
    for _ in range(args.warmup):
        time_oracle(w, inputs, rows, threads)
    total, flops = 0.0, 0.0
    for _ in range(args.steps):
        dt, f = time_oracle(w, inputs, rows, threads)
        total += dt
        flops += f
    value = flops / total / 1e12
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: Q, K, V iid N(0,1) fp32 rounded to bf16, seeded",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "seq_len": w.N, "parallelism": "host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{len(rows)} evenly spaced query rows per step of "
                                   f"{w.B * w.H * w.N} ({w.name}), fp64 C oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_seq_sharded(args, rank, world, local):
    """The workload's keys split over the ranks: a step is this rank's partial
    forward over its key shard, the all-gather of every rank's partial (O, LSE)
    and their merge; timed with CUDA events around whole steps, max over ranks."""
    import exact_attention_32_gb300 as fa
    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", local if world > 1 else 0)
    fa.lib()
    q_h, k_h, v_h = workload_inputs(w)
    begin, count = fa.fa_kv_shard(w.N, world, rank)
    q = q_h.to(dev)
    ks = k_h[:, :, begin:begin + count].contiguous().to(dev) if count else None
    vs = v_h[:, :, begin:begin + count].contiguous().to(dev) if count else None
    group = None
    if world > 1:
        import torch.distributed as dist
        group = dist.group.WORLD
    stream = torch.cuda.current_stream(dev)
    part_ms = []

    def step(record=False):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        o_part, lse_part = fa.forward_kv_shard(q, ks, vs, rank, world, scale=w.scale, causal=w.causal,
                                               stream=stream)
        e1.record(stream)
        if world > 1:
            o_parts, lse_parts = fa.gather_parts(o_part, lse_part, group)
        else:
            o_parts, lse_parts = o_part.unsqueeze(0), lse_part.unsqueeze(0)
        out = fa.combine(o_parts, lse_parts, stream=stream)
        if record:
            part_ms.append((e0, e1))
        return out

    for _ in range(args.warmup):
        step()
    K = args.steps
    clocks = ClockSampler(dev.index) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        step(record=True)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop() if clocks else None
    st = fa.fa_get_device_status(stream.cuda_stream)
    if st != 0:
        raise fa.FAError(st, "sequence-sharded step")
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    if rank != 0:
        return None
    part = statistics.mean(a.elapsed_time(b) for a, b in part_ms)  # rank 0's partial forward
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    # rank 0's partial forward: its keys against every query (causal: the
    # admitted pairs only; rank 0's shard has the most)
    lo, n = fa.fa_kv_shard(w.N, world, 0)
    pairs = sum(min(n, max(0, i + 1 - lo)) for i in range(w.N)) if w.causal else w.N * n
    part_flops = 4.0 * w.B * w.H * pairs * w.d
    value = w.flops * K / (total_ms / 1e3) / 1e12
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: Q, K, V iid N(0,1) fp32 rounded to bf16, seeded",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "scale": w.scale, "global_batch": w.B, "seq_len": w.N, "parallelism": f"kv_shards{world}",
                   "shard_rank0": {"begin": lo, "count": n},
                   "step": "fa_fwd_kv_shard + all-gather of (O, LSE) parts + fa_combine"},
        "roofline": {"bound": "tensor", "kernel": "fa_fwd_tc_kernel (key-shard partial)",
                     "achieved": part_flops / (part / 1e3) / 1e12, "peak": peak,
                     "peak_source": f"{peak_src} bf16_tflops (burst)", "unit": "TFLOP/s",
                     "frac": part_flops / (part / 1e3) / 1e12 / peak, "traffic": None,
                     "algorithmic_flops_per_launch": part_flops, "launch_ms": part},
        "gpu_launches": 2 * K,
        "clocks": clk,
        "impl": "ours",
    }


def main():
    args = parse_args()
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.shard == "seq":
        line = run_seq_sharded(args, rank, world, local)
    else:
        line = run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
