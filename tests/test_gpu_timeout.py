"""A bounded device-side wait that runs out (GPU).

The GQA kernel's producer warp feeds the consumer warps through
shared-memory stages that complete on mbarrier transaction counts, and the
dynamic-FP8 latent gather's warps feed themselves the same way; every wait is
bounded and, when the bound is reached, the kernel sets KVW_ERR_TIMEOUT,
gives up its work and returns instead of hanging.

To make a wait run out without faulting anything, the kernel source is
compiled a second time with -DKVW_TEST_HOOKS into a library of this test's
own (the product library has no such entry point).  Its GQA entry point
announces the first group of every CTA on that stage's barrier but never
issues the copies, so the consumers' wait for the stage can only end at its
limit (a few milliseconds here); its gather entry point does the same with
the first step of every warp.  The test checks that the call returns, the
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


def _hook_library(tmp_path_factory, source):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_kv_cache_mla_gb300 import build

    out = str(tmp_path_factory.mktemp("hooks") / ("libkvw_testhooks_" + source[:-3] + ".so"))
    cmd = [build.nvcc(), *build.ARCH, *build.NVCC_FLAGS, "-I", CSRC, "-DKVW_TEST_HOOKS",
           "-shared", "-cudart", "static", os.path.join(CSRC, source), "-o", out]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return ctypes.CDLL(out)


@pytest.fixture(scope="module")
def hooks(tmp_path_factory):
    L = _hook_library(tmp_path_factory, "qk_rope_paged_ragged.cu")
    vp, u32 = ctypes.c_void_p, ctypes.c_uint32
    from gqa_kv_cache_mla_gb300 import kvw

    f = L.kvw_test_qk_rope_withheld_stage
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, u32, u32, u32, ctypes.POINTER(kvw.PagedCacheT), vp, u32, vp,
                  ctypes.c_int, u32, vp, vp, vp, ctypes.c_uint64]
    return f


@pytest.fixture(scope="module")
def gather_hooks(tmp_path_factory):
    L = _hook_library(tmp_path_factory, "mla_gather_latent.cu")
    vp, u32 = ctypes.c_void_p, ctypes.c_uint32
    from gqa_kv_cache_mla_gb300 import kvw

    f = L.kvw_test_gather_dynamic_withheld_stage
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, ctypes.POINTER(kvw.PagedCacheT), u32, vp, u32, u32, vp, vp,
                  ctypes.c_uint64]
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



@pytest.mark.parametrize("cache_dtype", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
def test_gather_withheld_stage_times_out_and_returns(orc, dev, gather_hooks, cache_dtype):
    import torch

    # 20,171 rows: 5,043 warp steps of 4 rows, more than the warps of one
    # wave (152 SMs x 3 CTAs x 8 warps on a GB300), so many warps also have a
    # second, normally copied stage in flight to wait for before they return
    w = W.mla_workload("tg", 1311, [3, 0, 17, 1, 40, 70], [5000, 9, 8000, 31, 0, 7000],
                       num_heads=1, page_size=16, max_seq_len=8192, cache_dtype=cache_dtype,
                       num_layers=2, layer_idx=1)
    g = W.mla_gather(w, dynamic=True)
    d = dev.DeviceGather(g)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert gather_hooks(d.out.tensor.data_ptr(), d.scales.tensor.data_ptr(), ctypes.byref(d.desc),
                        g.layer_idx, d.ctx.tensor.data_ptr(), g.ctx_offsets.shape[0] - 1, g.rows,
                        d.err.tensor.data_ptr(), ctypes.c_void_p(stream.cuda_stream),
                        WAIT_NS) == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0, elapsed
    assert d.flags() & KVW_ERR_TIMEOUT
    assert d.guards_intact()
    assert np.array_equal(d.cache.host(), g.cache.data)
    assert np.array_equal(d.out.host(), d.out_init)  # every warp gave up at its first step
    assert not d.scales.host().any()

    # the context is still usable: the product entry point on the same inputs
    d.clear_flags()
    d.run()
    torch.cuda.synchronize()
    ref, ref_scales, f_ref = orc.mla_gather_latent_dynamic(
        g.cache, g.layer_idx, g.ctx_offsets, out=d.out_init.copy(),
        scales=np.zeros(g.rows, np.float32))
    assert d.flags() == f_ref == 0
    assert np.array_equal(d.scales.host(), ref_scales)
    assert np.array_equal(d.out.host(), ref)
