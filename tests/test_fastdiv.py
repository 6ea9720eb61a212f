"""Host check of the multiply-shift division used by the kernels (CPU only):
compiles a small host program against csrc/common.cuh and compares with
integer division for divisors 1..4999 and a set of large ones."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fastdiv_matches_integer_division(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "fastdiv_check"
    subprocess.run([nvcc, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "bwd_maxpool3d_fwd_gb300", "csrc"),
                    "-o", str(exe), os.path.join(ROOT, "tests", "fastdiv_check.cu")], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    assert "bad=0" in out.stdout
