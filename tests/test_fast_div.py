"""Division by a run-time invariant (FastDiv in the kernels' device header)
against the hardware division, compiled and run on the host (tests/c/fast_div.cu):
every divisor 1..70000 at the numerators around its multiples and the ends of
the 32-bit range, and 2e7 pseudo-random pairs."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fast_div_matches_division(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    exe = str(tmp_path / "fast_div")
    subprocess.run([nvcc, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(ROOT, "gqa_kv_cache_mla_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "c", "fast_div.cu"), "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert " 0 wrong" in r.stdout
