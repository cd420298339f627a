"""A bounded device-side wait that runs out (GPU).

The GQA kernel's producer warp feeds the consumer warps through
shared-memory stages that complete on mbarrier transaction counts; every
wait is bounded and, when the bound is reached, the kernel sets
KVW_ERR_TIMEOUT, gives up its work and returns instead of hanging.

To make a wait run out without faulting anything, the kernel source is
compiled a second time with -DKVW_TEST_HOOKS into a library of this test's
own (the product library has no such entry point).  Its entry point
announces the first group of every CTA on that stage's barrier but never
issues the copies, so the consumers' wait for the stage can only end at its
limit (a few milliseconds here).  The test checks that the call returns, the
flag is set, no byte of the cache or of the output changed (the consumers
gave up before writing anything), the guard bytes around every buffer are
intact, and that the context is still usable: the product entry point then
matches the CPU reference on the same inputs.
"""
import ctypes
import os
import subprocess
import time

import numpy as np
import pytest

from gqa_kv_cache_mla_gb300 import workloads as W
from helpers import compare_bf16, compare_cache, expected_slots

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gqa_kv_cache_mla_gb300", "csrc")
KVW_ERR_TIMEOUT = 8
WAIT_NS = 2_000_000  # 2 ms


@pytest.fixture(scope="module")
def hooks(tmp_path_factory):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_kv_cache_mla_gb300 import build

    out = str(tmp_path_factory.mktemp("hooks") / "libkvw_testhooks.so")
    cmd = [build.nvcc(), *build.ARCH, *build.NVCC_FLAGS, "-I", CSRC, "-DKVW_TEST_HOOKS",
           "-shared", "-cudart", "static", os.path.join(CSRC, "qk_rope_paged_ragged.cu"),
           "-o", out]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    L = ctypes.CDLL(out)
    vp, u32 = ctypes.c_void_p, ctypes.c_uint32
    from gqa_kv_cache_mla_gb300 import kvw

    f = L.kvw_test_qk_rope_withheld_stage
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, u32, u32, u32, ctypes.POINTER(kvw.PagedCacheT), vp, u32, vp,
                  ctypes.c_int, u32, vp, vp, vp, ctypes.c_uint64]
    return f


@pytest.fixture(scope="module")
def dev():
    from gqa_kv_cache_mla_gb300 import device

    return device


def _withheld_call(hooks, d, w, wait_ns):
    import torch

    stream = torch.cuda.current_stream()
    return hooks(d.q.tensor.data_ptr(), d.offsets.tensor.data_ptr(), w.B, w.T,
                 w.q_proj.shape[1], ctypes.byref(d.desc), d.freqs.tensor.data_ptr(),
                 w.freqs.shape[0],
                 None if d.pos is None else d.pos.tensor.data_ptr(), int(w.interleaved),
                 w.layer_idx, d.out.tensor.data_ptr(), d.err.tensor.data_ptr(),
                 ctypes.c_void_p(stream.cuda_stream), wait_ns)


@pytest.mark.parametrize("cache_dtype,interleaved,mode",
                         [(W.DTYPE_BF16, True, None), (W.DTYPE_FP8_E4M3, False, "ids")])
def test_withheld_stage_times_out_and_returns(orc, dev, hooks, cache_dtype, interleaved, mode):
    import torch

    # 1,904 tokens: more groups than CTAs, so some CTAs also wait for a free
    # stage (which never comes) after their withheld first group
    w = W.gqa_workload("to", 1301, [400, 3, 1500, 1], [0, 250, 9, 31], 8, 2, 128,
                       page_size=32, freqs_rows=2048, base=500000.0, interleaved=interleaved,
                       position_mode=mode, cache_dtype=cache_dtype)
    d = dev.DeviceGQA(w)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _withheld_call(hooks, d, w, WAIT_NS) == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0, elapsed
    assert d.flags() & KVW_ERR_TIMEOUT
    assert d.guards_intact()
    assert np.array_equal(d.cache.host(), w.cache.data)
    assert np.array_equal(d.out.host(), d.out_init)

    # the context is still usable: the product entry point on the same inputs
    d.clear_flags()
    d.run()
    torch.cuda.synchronize()
    out_ref, c_ref, f_ref = orc.qk_rope_paged_ragged(w, output=d.out_init.copy())
    assert d.flags() == f_ref == 0
    compare_bf16(d.out.host(), out_ref)
    c = w.cache
    compare_cache(c, d.cache.host(), c_ref,
                  expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size),
                  w.layer_idx, fp8=cache_dtype == W.DTYPE_FP8_E4M3)

