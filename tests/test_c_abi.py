"""The C ABI from a plain C program (tests/c/abi_mla.c): it compiles and links
against the library and the CPU reference everywhere, and on a GPU it runs the
fused MLA write on a small ragged batch and matches the reference."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build(tmp_path):
    import oracle
    from gqa_kv_cache_mla_gb300 import kvw

    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    oracle.build()
    libdirs = [os.path.dirname(kvw.LIB_PATH), os.path.join(ROOT, "oracle")]
    exe = str(tmp_path / "abi_mla")
    cmd = [nvcc, os.path.join(ROOT, "tests", "c", "abi_mla.c"),
           "-I", os.path.join(ROOT, "include"), "-o", exe, "-lkvw", "-loracle", "-lm"]
    for d in libdirs:
        cmd += ["-L", d, "-Xlinker", "-rpath=" + d]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_program_builds_against_the_header(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
@pytest.mark.parametrize("cache_dtype", [0, 1])
def test_c_program_matches_the_reference(tmp_path, cache_dtype):
    exe = _build(tmp_path)
    r = subprocess.run([exe, str(cache_dtype)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 mismatches" in r.stdout
