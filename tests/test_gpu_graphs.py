"""Every entry point captured into a CUDA graph and replayed (GPU).

The library's calls are asynchronous on the stream they are given, allocate
nothing and read nothing back to the host, so a serving loop can capture a
step's calls once and replay the graph.  Each case here makes one ordinary
call first (as the loop's first step would: the per-device launch facts are
cached then), puts every device buffer back to its initial bytes, captures
one call on a side stream, restores the buffers again and replays the
graph once; the result must be the oracle's, compared exactly as the parity
tests compare a direct call.
"""
import numpy as np
import pytest

from gqa_kv_cache_mla_gb300 import workloads as W
from test_gpu_parity import run_gather, run_gqa, run_knorm, run_mla

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_kv_cache_mla_gb300 import device

    return device


def in_graph(d, **kw):
    """Capture one call of `d`'s entry point into a CUDA graph and replay it
    on the initial buffer contents."""
    import torch

    initial = [(b, b.host().copy()) for b in d.buffers]

    def restore():
        for b, h in initial:
            b.reset(h)
        torch.cuda.synchronize()

    d.run(**kw)
    torch.cuda.synchronize()
    restore()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        d.run(stream=s, **kw)
    torch.cuda.synchronize()
    restore()
    g.replay()
    torch.cuda.synchronize()
    assert g is not None


def _mla(cache_dtype, **kw):
    return W.mla_workload("gr", 1401, [3, 0, 17, 1, 40], [5, 9, 100, 31, 0], num_heads=8,
                          page_size=16, max_seq_len=256, cache_dtype=cache_dtype, num_layers=2,
                          layer_idx=1, **kw)


@pytest.mark.parametrize("cache_dtype", [W.DTYPE_FP8_E4M3, W.DTYPE_BF16])
def test_mla_quant_in_graph(orc, dev, cache_dtype):
    run_mla(orc, dev, _mla(cache_dtype), launch=in_graph)


def test_mla_decode_fast_path_in_graph(orc, dev):
    w = W.mla_workload("grd", 1402, np.ones(40, np.int64), np.arange(40) * 7, num_heads=16,
                       page_size=16, max_seq_len=512, cache_dtype=W.DTYPE_FP8_E4M3)
    run_mla(orc, dev, w, launch=in_graph)


def test_mla_inplace_and_fp8_q_in_graph(orc, dev):
    run_mla(orc, dev, W.mla_inplace(_mla(W.DTYPE_BF16)), launch=in_graph)
    w = _mla(W.DTYPE_FP8_E4M3)
    w.q_out_dtype = W.DTYPE_FP8_E4M3
    run_mla(orc, dev, w, launch=in_graph)


@pytest.mark.parametrize("mode,cache_dtype", [(None, W.DTYPE_BF16), ("ids", W.DTYPE_FP8_E4M3),
                                              ("mrope", W.DTYPE_BF16)])
def test_gqa_in_graph(orc, dev, mode, cache_dtype):
    w = W.gqa_workload("gr", 1403, [3, 17, 1, 200], [0, 40, 300, 9], 8, 2, 128, page_size=16,
                       freqs_rows=1024, base=500000.0, interleaved=mode != "ids",
                       position_mode=mode,
                       mrope_section=(16, 24, 24) if mode == "mrope" else None,
                       cache_dtype=cache_dtype)
    run_gqa(orc, dev, w, launch=in_graph)


@pytest.mark.parametrize("gamma_len,per_head", [(128, True), (64, True), (96, True),
                                                (256, False)])
def test_knorm_in_graph(orc, dev, gamma_len, per_head):
    w = W.knorm_workload("gr", 1404, [3, 17, 1, 200], [0, 40, 300, 9], 2, 128, page_size=16,
                         gamma_len=gamma_len)
    run_knorm(orc, dev, w, per_head_norm=per_head, launch=in_graph)


@pytest.mark.parametrize("dynamic", [False, True])
def test_gather_in_graph(orc, dev, dynamic):
    run_gather(orc, dev, W.mla_gather(_mla(W.DTYPE_BF16), dynamic=dynamic), launch=in_graph)


@pytest.mark.parametrize("per_row", [False, True])
def test_fp8_codecs_in_graph(orc, dev, per_row):
    rng = np.random.default_rng(1405)
    if per_row:
        w = W.ConvertWorkload("gr", W.normal_bf16(rng, (300, 1000)), 1.0, per_row=True)
    else:
        w = W.ConvertWorkload("gr", W.normal_bf16(rng, (1 << 16,), std=0.05), 0.5)
    d = dev.DeviceConvert(w)
    in_graph(d)
    assert d.guards_intact()
    if per_row:
        codes, scales = orc.quantize_rows_e4m3(w.x)
        assert np.array_equal(d.scales.host(), scales) and np.array_equal(d.out.host(), codes)
    else:
        assert np.array_equal(d.out.host(), orc.convert_bf16_to_e4m3(w.x, w.scale))
