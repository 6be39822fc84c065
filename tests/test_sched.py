"""The Stream-K partition of the GEMM kernels, checked on the CPU: the kernel header's scheduling code compiled for the
host (tests/sched_check.cu) covers every (tile, K block) exactly once and the split-K reduction reads exactly the
partial slots the GEMM writes."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_stream_k_partition(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = tmp_path / "sched_check"
    subprocess.run([nvcc, "-std=c++17", "-O2", "--expt-relaxed-constexpr", "-o", str(exe), os.path.join(HERE, "sched_check.cu")], check=True,
                   capture_output=True, timeout=600)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.startswith("OK"), r.stdout[-2000:]
