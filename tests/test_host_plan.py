"""Host check of the packed layout and the GEMV work plans (CPU only).

Compiles tests/host/plan_walk.cpp with the library's packer and planners
against a stub CUDA runtime (device memory is host memory) and runs it. The
program replays every warp's walk of the batch-1 kernels over seeded matrices.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mixed_precision_weight_bit_b300", "csrc")


def test_plan_walk(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "plan_walk")
    cmd = [cxx, "-O2", "-std=c++17", "-I/usr/local/cuda/include", os.path.join(ROOT, "tests", "host", "plan_walk.cpp"),
           os.path.join(CSRC, "pack.cpp"), os.path.join(CSRC, "plan.cpp"), os.path.join(CSRC, "gemv_plan.cpp"), "-o", exe, "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "plan walk ok" in r.stdout
