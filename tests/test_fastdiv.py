"""The kernels' division by invariant divisors (split_gemm_gb300/csrc/fastdiv.h) against
plain integer division over every divisor shape the launch parameters take (CPU only)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fastdiv_matches_integer_division(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = tmp_path / "fastdiv_check"
    src = os.path.join(ROOT, "tests", "c", "fastdiv_check.cpp")
    inc = os.path.join(ROOT, "split_gemm_gb300", "csrc")
    subprocess.run([gxx, "-std=c++17", "-O2", "-I", inc, src, "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "0 wrong" in res.stdout
