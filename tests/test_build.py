"""Sources that only the GPU tests build still compile here (nvcc cross-compiles
for sm_103a without a device), so a change to the shared headers that breaks
them fails the CPU suite rather than the GPU one."""
import os
import shutil
import subprocess
import tempfile

import pytest

from exact_attention_32_gb300 import build as fa_build

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tcgen05_selftest_source_compiles():
    try:
        nvcc = fa_build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    out = tempfile.mkdtemp()
    try:
        r = subprocess.run([nvcc] + fa_build.ARCH +
                           ["-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-c", "-I", fa_build.CSRC,
                            os.path.join(HERE, "cuda", "tc_selftest.cu"), "-o", os.path.join(out, "t.o")],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
    finally:
        shutil.rmtree(out, ignore_errors=True)
