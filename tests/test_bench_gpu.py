"""bench.py on the GPU: the default step and the sequence-sharded step each
print one JSON line of the contract's shape on a small workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def run_bench(*extra):
    cmd = [sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--no-e2e", "--no-cpu-baseline",
           "--no-secondary", "--workload", "b16_h16_n1000_d64_causal_q8", *extra]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_default_step_line():
    d = run_bench()
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["value"] > 0 and d["gpu_launches"] == 3
    assert d["roofline"]["kernel"] == "fa_fwd_dp_kernel" and 0 < d["roofline"]["frac"] < 1.5
    assert d["config"]["parallelism"] == "bh_slabs1"


def test_sequence_sharded_step_line():
    d = run_bench("--shard", "seq")
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["value"] > 0 and d["gpu_launches"] == 6
    assert d["scaling"] == "strong" and d["config"]["parallelism"] == "kv_shards1"
    assert d["config"]["shard_rank0"] == {"begin": 0, "count": 1000}
    assert 0 < d["roofline"]["frac"] < 1.5
