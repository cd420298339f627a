import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


def _build_library():
    """Compile libkvw.so (host-side checks and the ABI tests load it) and the oracle."""
    import shutil

    if shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc"):
        from gqa_kv_cache_mla_gb300 import build

        build.build()


_build_library()
