"""Host logic: the split-KV work schedule, compiled from the same header the
kernels use (nvcc, host code only) and walked on the CPU."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


@pytest.mark.skipif(not os.path.exists(NVCC), reason="nvcc not available")
def test_schedule_walk(tmp_path):
    exe = tmp_path / "schedule_check"
    r = subprocess.run([NVCC, "-std=c++17", "-O1", "-o", str(exe),
                        os.path.join(HERE, "schedule_check.cu")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK")
