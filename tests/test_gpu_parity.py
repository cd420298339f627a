"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every case builds a seeded workload, runs the oracle on the host and the
kernel on the device on the same bytes, and compares element by element:
  * bytes outside the rows a call may write: bit-identical (guard bytes
    around every device buffer included);
  * bf16 outputs: at most 1 bf16 ulp from the oracle's fp32 result rounded
    to bf16;
  * FP8 E4M3 cache values: at most 1 E4M3 ulp on at most 0.1% of the written
    elements (scale convention: stored = satfinite_rne(y / scale));
  * error flags: equal.
The five benchmark workloads run at full size in the launch configuration
the benchmark uses; small cases cover edges.
"""
import os

import numpy as np
import pytest

from gqa_kv_cache_mla_gb300 import workloads as W
from helpers import compare_bf16, compare_cache, compare_e4m3, expected_slots

pytestmark = pytest.mark.gpu

NTHREADS = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


@pytest.fixture(scope="module")
def dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_kv_cache_mla_gb300 import device

    return device


def _launch(d, **kw):
    """One call of the entry point a device holder wraps, on the current stream."""
    d.run(**kw)


def run_mla(orc, dev, w, launch=None, **kw):
    d = dev.DeviceMLA(w)
    (launch or _launch)(d)
    import torch

    torch.cuda.synchronize()
    fn = orc.mla_rope_rmsnorm_inplace if w.inplace else orc.mla_rope_rmsnorm_quant
    q_ref, c_ref, f_ref = fn(w, q_rope_out=d.q_out_init.copy(), nthreads=NTHREADS,
                             out_dtype=w.q_out_dtype)
    assert d.guards_intact()
    assert d.flags() == f_ref
    c = w.cache
    if w.q_out_dtype == W.DTYPE_BF16:
        nq = compare_bf16(d.q_out.host(), q_ref)
    else:
        nq = compare_e4m3(d.q_out.host(), q_ref)
    slots = [] if f_ref & 4 else expected_slots(w.offsets, c.cache_lengths, c.page_table,
                                                c.page_size, c.num_pages)
    nc = compare_cache(c, d.cache.host(), c_ref, slots, w.layer_idx,
                       fp8=c.dtype == W.DTYPE_FP8_E4M3)
    return d, nq, nc


# ------------------------------------------------------------------ MLA

@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
def test_mla_tiny(orc, dev, dtype):
    run_mla(orc, dev, W.mla_tiny(cache_dtype=dtype))


@pytest.mark.parametrize("dtype", [W.DTYPE_FP8_E4M3, W.DTYPE_BF16])
def test_mla_decode_full(orc, dev, dtype):
    run_mla(orc, dev, W.mla_decode(cache_dtype=dtype))


@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
def test_mla_prefill_full(orc, dev, dtype):
    run_mla(orc, dev, W.mla_prefill(cache_dtype=dtype))


@pytest.mark.parametrize("H", [0, 1, 3, 16, 33])
def test_mla_head_counts_and_ragged_tail(orc, dev, H):
    w = W.mla_workload("h", 200 + H, [1, 0, 37, 5, 130], [3, 9, 0, 250, 17], num_heads=H,
                       page_size=16, max_seq_len=512, cache_dtype=W.DTYPE_FP8_E4M3,
                       num_layers=3, layer_idx=2, spare_pages=3)
    run_mla(orc, dev, w)


def test_mla_strided_kv_rows(orc, dev):
    w = W.mla_workload("s", 211, [7, 9], [0, 100], num_heads=8, page_size=32, max_seq_len=256,
                       cache_dtype=W.DTYPE_BF16)
    rng = np.random.default_rng(5)
    wide = rng.integers(0, 2**16, size=(w.T, 640), dtype=np.uint16)
    wide[:, 64:640] = w.kv_in  # the 576-wide rows sit at column 64 of a 640-wide buffer
    d = dev.DeviceMLA(w)
    import torch

    buf = torch.from_numpy(wide.view(np.int16)).to("cuda")
    from gqa_kv_cache_mla_gb300 import kvw

    kvw.kvw_mla_rope_rmsnorm_quant(d.q_out.tensor, d.q.tensor, d.offsets.tensor, d.freqs.tensor,
                                   d.gamma.tensor, buf[:, 64:], d.desc, w.layer_idx, w.epsilon,
                                   d.err.tensor, kv_row_stride=640)
    torch.cuda.synchronize()
    q_ref, c_ref, f = orc.mla_rope_rmsnorm_quant(w, q_rope_out=d.q_out_init.copy())
    c = w.cache
    compare_bf16(d.q_out.host(), q_ref)
    compare_cache(c, d.cache.host(), c_ref,
                  expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size),
                  w.layer_idx, fp8=False)


def test_mla_many_requests_and_page_size_one(orc, dev):
    rng = np.random.default_rng(7)
    B = 3000
    new = rng.integers(0, 3, B)
    prior = rng.integers(0, 60, B)
    w = W.mla_workload("m", 212, new, prior, num_heads=2, page_size=1, max_seq_len=64,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    run_mla(orc, dev, w)


@pytest.mark.parametrize("kind", ["gqa", "gqa_fp8k", "gqa_mrope", "knorm64", "knorm_row",
                                  "gather", "gather_dynamic"])
def test_page_size_one(orc, dev, kind):
    """Pages of one token: every row of a request sits on its own page, so
    consecutive rows are never adjacent and every slot lookup is distinct."""
    rng = np.random.default_rng(1501)
    B = 300
    new = rng.integers(0, 4, B)
    prior = rng.integers(0, 40, B)
    if kind.startswith("gqa"):
        mode = "mrope" if kind == "gqa_mrope" else None
        w = W.gqa_workload("p1", 1502, new, prior, 8, 2, 64, page_size=1, freqs_rows=64,
                           base=10000.0, interleaved=kind != "gqa_mrope", position_mode=mode,
                           mrope_section=(8, 12, 12) if mode else None,
                           cache_dtype=W.DTYPE_FP8_E4M3 if kind == "gqa_fp8k" else W.DTYPE_BF16)
        run_gqa(orc, dev, w)
    elif kind.startswith("knorm"):
        per_head = kind == "knorm64"
        w = W.knorm_workload("p1", 1503, new, prior, 2, 128, page_size=1,
                             gamma_len=64 if per_head else 256)
        run_knorm(orc, dev, w, per_head_norm=per_head)
    else:
        w = W.mla_workload("p1", 1504, new, prior, num_heads=1, page_size=1, max_seq_len=64,
                           cache_dtype=W.DTYPE_BF16)
        run_gather(orc, dev, W.mla_gather(w, dynamic=kind == "gather_dynamic"))


@pytest.mark.parametrize("page", [3, 12, 48, 100])
@pytest.mark.parametrize("kind", ["mla", "gqa", "knorm", "gather_dynamic"])
def test_page_sizes_not_powers_of_two(orc, dev, kind, page):
    """Page sizes with no power-of-two factor to shift by: the kernels divide
    slot positions by the page size through multiply-high constants, which
    must give the exact quotient and remainder for every position."""
    rng = np.random.default_rng(1600 + page)
    B = 40
    new = rng.integers(0, 40, B)
    prior = rng.integers(0, 400, B)
    max_seq = int(-(-int((new + prior).max() + 1) // page) * page)
    if kind == "mla":
        w = W.mla_workload("pp", 1601 + page, new, prior, num_heads=3, page_size=page,
                           max_seq_len=max_seq, cache_dtype=W.DTYPE_FP8_E4M3, num_layers=2,
                           layer_idx=1)
        run_mla(orc, dev, w)
    elif kind == "gqa":
        w = W.gqa_workload("pp", 1602 + page, new, prior, 8, 2, 128, page_size=page,
                           freqs_rows=max_seq, base=500000.0, interleaved=True)
        run_gqa(orc, dev, w)
    elif kind == "knorm":
        w = W.knorm_workload("pp", 1603 + page, new, prior, 3, 128, page_size=page,
                             gamma_len=64)
        run_knorm(orc, dev, w)
    else:
        w = W.mla_workload("pp", 1604 + page, new, prior, num_heads=1, page_size=page,
                           max_seq_len=max_seq, cache_dtype=W.DTYPE_BF16)
        run_gather(orc, dev, W.mla_gather(w, dynamic=True))


def test_mla_error_flags(orc, dev):
    # position past the table
    w = W.mla_workload("p", 91, [2, 5], [0, 60], num_heads=2, page_size=16, max_seq_len=80,
                       cache_dtype=W.DTYPE_BF16)
    w.freqs = w.freqs[:64].copy()
    d, _, _ = run_mla(orc, dev, w)
    assert d.flags() == 2
    # unmapped page
    w = W.mla_tiny()
    w.cache.page_table[1, 0] = W.PAGE_UNMAPPED
    d, _, _ = run_mla(orc, dev, w)
    assert d.flags() == 1
    # bad offsets: nothing written
    for bad in ([1, 3, 8], [0, 5, 3, 8], [0, 3, 7]):
        w = W.mla_tiny()
        w.offsets = np.array(bad, np.uint32)
        d = dev.DeviceMLA(w)
        d.run(tot_seq_len=8)
        import torch

        torch.cuda.synchronize()
        assert d.flags() == 4
        assert np.array_equal(d.cache.host(), w.cache.data)
        assert np.array_equal(d.q_out.host(), d.q_out_init)


def test_mla_empty_and_repeat(orc, dev):
    import torch

    w = W.mla_workload("e", 93, [0, 0], [3, 0], num_heads=2, page_size=16, max_seq_len=32,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    d = dev.DeviceMLA(w)
    d.run()
    torch.cuda.synchronize()
    assert d.flags() == 0 and np.array_equal(d.cache.host(), w.cache.data)
    # two identical calls give identical bytes
    w = W.mla_tiny(cache_dtype=W.DTYPE_FP8_E4M3)
    d = dev.DeviceMLA(w)
    d.run()
    torch.cuda.synchronize()
    a = (d.q_out.host().copy(), d.cache.host().copy())
    d.cache.reset(w.cache.data)
    s = torch.cuda.Stream()
    d.run(stream=s)
    s.synchronize()
    assert np.array_equal(a[0], d.q_out.host()) and np.array_equal(a[1], d.cache.host())


# ------------------------------------------------- MLA decode batches (T == B)
# With as many tokens as requests the kernel first assumes the offsets are
# the identity (one token per request) and verifies that over the whole
# table; any other table takes the general path.  Both must give the
# oracle's results and flags.

@pytest.mark.parametrize("B,H", [(1, 128), (5, 3), (13, 1), (700, 2), (300, 0)])
@pytest.mark.parametrize("dtype", [W.DTYPE_FP8_E4M3, W.DTYPE_BF16])
def test_mla_decode_identity_shapes(orc, dev, B, H, dtype):
    rng = np.random.default_rng(1000 + B + H)
    prior = rng.integers(0, 900, B)
    w = W.mla_workload("dec", 1001 + B, np.ones(B, np.int64), prior, num_heads=H,
                       page_size=16, max_seq_len=1024, cache_dtype=dtype, num_layers=2,
                       layer_idx=1)
    run_mla(orc, dev, w)


@pytest.mark.parametrize("variant", ["inplace", "fp8q"])
def test_mla_decode_identity_variants(orc, dev, variant):
    rng = np.random.default_rng(1010)
    B = 37
    w = W.mla_workload("decv", 1011, np.ones(B, np.int64), rng.integers(0, 500, B),
                       num_heads=5, page_size=32, max_seq_len=512,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    if variant == "inplace":
        w = W.mla_inplace(w)
    else:
        w.q_out_dtype = W.DTYPE_FP8_E4M3
    run_mla(orc, dev, w)


def test_mla_decode_count_but_not_identity(orc, dev):
    # T == B, valid offsets, but requests with 0 and 2+ new tokens
    new = np.array([2, 0, 1, 1, 3, 0, 0, 1])
    w = W.mla_workload("dni", 1021, new, [5, 0, 17, 3, 40, 9, 0, 2], num_heads=3,
                       page_size=16, max_seq_len=128, cache_dtype=W.DTYPE_FP8_E4M3)
    assert w.T == w.B
    run_mla(orc, dev, w)


def test_mla_decode_identity_flags(orc, dev):
    import torch

    B = 40
    prior = np.arange(B) * 3
    # positions past the table for the last requests
    w = W.mla_workload("dfp", 1031, np.ones(B, np.int64), prior, num_heads=4, page_size=16,
                       max_seq_len=128, cache_dtype=W.DTYPE_BF16)
    w.freqs = w.freqs[:100].copy()
    d, _, _ = run_mla(orc, dev, w)
    assert d.flags() == 2
    # an unmapped page
    w = W.mla_workload("dfg", 1032, np.ones(B, np.int64), prior, num_heads=4, page_size=16,
                       max_seq_len=128, cache_dtype=W.DTYPE_FP8_E4M3)
    w.cache.page_table[7, prior[7] // 16] = W.PAGE_UNMAPPED  # the page of request 7's token
    d, _, _ = run_mla(orc, dev, w)
    assert d.flags() == 1
    # T == B but the offsets are not a valid table: nothing is written
    for bad in ([0, 1, 1, 0, 4], [0, 1, 2, 3, 5], [1, 1, 2, 3, 4]):
        w = W.mla_workload("dbo", 1033, np.ones(4, np.int64), [3, 1, 4, 1], num_heads=2,
                           page_size=16, max_seq_len=64, cache_dtype=W.DTYPE_FP8_E4M3)
        w.offsets = np.array(bad, np.uint32)
        d = dev.DeviceMLA(w)
        d.run(tot_seq_len=4)
        torch.cuda.synchronize()
        assert d.flags() == 4
        assert np.array_equal(d.cache.host(), w.cache.data)
        assert np.array_equal(d.q_out.host(), d.q_out_init)


# ------------------------------------------------------------------ GQA

def run_gqa(orc, dev, w, alias=False, launch=None):
    import torch

    d = dev.DeviceGQA(w, alias_output=alias)
    (launch or _launch)(d)
    torch.cuda.synchronize()
    out0 = w.q_proj.copy() if alias else d.out_init.copy()
    if alias:
        w2 = W.GQAWorkload(**{**w.__dict__})
        w2.q_proj = out0
        out_ref, c_ref, f_ref = orc.qk_rope_paged_ragged(w2, output=out0, nthreads=NTHREADS)
    else:
        out_ref, c_ref, f_ref = orc.qk_rope_paged_ragged(w, output=out0, nthreads=NTHREADS)
    assert d.guards_intact()
    assert d.flags() == f_ref
    c = w.cache
    compare_bf16(d.out.host(), out_ref)
    slots = [] if f_ref & 4 else expected_slots(w.offsets, c.cache_lengths, c.page_table,
                                                c.page_size, c.num_pages)
    compare_cache(c, d.cache.host(), c_ref, slots, w.layer_idx,
                  fp8=c.dtype == W.DTYPE_FP8_E4M3)
    return d


@pytest.mark.parametrize("interleaved", [True, False])
@pytest.mark.parametrize("mode", [None, "ids", "mrope"])
def test_gqa_fp8_k_cache_full(orc, dev, interleaved, mode):
    run_gqa(orc, dev, W.gqa_llama3(interleaved=interleaved, position_mode=mode,
                                   cache_dtype=W.DTYPE_FP8_E4M3))


@pytest.mark.parametrize("scale", [0.5, 3.0])
@pytest.mark.parametrize("mode", [None, "mrope"])
def test_gqa_fp8_k_cache_scales_and_layouts(orc, dev, scale, mode):
    w = W.gqa_workload("f8", 730, [3, 0, 17, 1, 40], [0, 5, 100, 31, 7], 8, 4, 64, page_size=16,
                       freqs_rows=256, base=10000.0, interleaved=mode is None,
                       position_mode=mode, mrope_section=(5, 20, 7) if mode else None,
                       cache_dtype=W.DTYPE_FP8_E4M3, scale=scale)
    run_gqa(orc, dev, w)
    w.cache = W.repad_cache(w.cache, 16, 32)  # non-adjacent heads: per-head copies
    run_gqa(orc, dev, w)


@pytest.mark.parametrize("interleaved", [True, False])
@pytest.mark.parametrize("mode", [None, "ids", "mrope"])
def test_gqa_llama3_full(orc, dev, interleaved, mode):
    run_gqa(orc, dev, W.gqa_llama3(interleaved=interleaved, position_mode=mode))


@pytest.mark.parametrize("S,Hq,Hk,sec", [(64, 8, 2, (5, 20, 7)), (256, 4, 1, (40, 44, 44)),
                                         (16, 3, 1, (1, 3, 4)), (128, 64, 8, (16, 24, 24))])
@pytest.mark.parametrize("interleaved", [True, False])
def test_gqa_shapes_and_odd_sections(orc, dev, S, Hq, Hk, sec, interleaved):
    w = W.gqa_workload("s", 300 + S, [3, 0, 17, 1, 40], [0, 5, 100, 31, 7], Hq, Hk, S,
                       page_size=16, freqs_rows=256, base=10000.0, interleaved=interleaved,
                       position_mode="mrope", mrope_section=sec, spare_pages=2)
    run_gqa(orc, dev, w)
    w = W.gqa_workload("s", 400 + S, [3, 0, 17, 1, 40], [0, 5, 100, 31, 7], Hq, Hk, S,
                       page_size=16, freqs_rows=256, base=10000.0, interleaved=interleaved)
    run_gqa(orc, dev, w)


def test_gqa_output_aliases_input(orc, dev):
    w = W.gqa_workload("a", 501, [4, 9, 1], [3, 0, 20], 8, 2, 128, page_size=16,
                       freqs_rows=64, base=500000.0, interleaved=False, position_mode="ids")
    run_gqa(orc, dev, w, alias=True)


def test_gqa_error_flags(orc, dev):
    w = W.gqa_workload("g", 72, [3, 5], [0, 7], 2, 2, 16, page_size=16, freqs_rows=64,
                       base=10000.0, interleaved=True, position_mode="ids")
    w.position_ids[4] = 64
    w.cache.page_table[0, 0] = W.PAGE_UNMAPPED
    d = run_gqa(orc, dev, w)
    assert d.flags() == 3


# ------------------------------------------------------------------ K norm

def run_knorm(orc, dev, w, per_head_norm=True, launch=None):
    import torch

    d = dev.DeviceKNorm(w)
    (launch or _launch)(d, per_head_norm=per_head_norm)
    torch.cuda.synchronize()
    c_ref, f_ref = orc.rms_norm_kv_cache_paged(w, per_head_norm=per_head_norm, nthreads=NTHREADS)
    assert d.guards_intact()
    assert d.flags() == f_ref
    c = w.cache
    slots = [] if f_ref & 4 else expected_slots(w.offsets, c.cache_lengths, c.page_table,
                                                c.page_size, c.num_pages)
    compare_cache(c, d.cache.host(), c_ref, slots, w.layer_idx, fp8=False,
                  cols=w.gamma.size if per_head_norm else None,
                  bf16_max_ulp=1 if w.multiply_before_cast else knorm_cast_first_ulp(w))
    return d


def knorm_cast_first_ulp(w):
    """Tolerance of multiply_before_cast=false, which rounds twice: y1 = bf16(x*r),
    then bf16(y1*wt) with wt = gamma + weight_offset.  The kernel sums the
    squares in another order and refines an rsqrt estimate of 1/rms, so r can
    differ in its last fp32 bits and y1 by one bf16 ulp u1; the products then differ by |wt|*u1.  For |wt| >= 1 the
    result's ulp is at least u1 (and at least |wt|*u1/2), so the exact products
    differ by less than 2 result ulps and the rounded ones by at most 2; for
    |wt| < 1 the result's ulp can be as small as |wt|*u1/2, giving at most 3."""
    g = (w.gamma.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return 2 if np.abs(g + w.weight_offset).min() >= 1.0 else 3


@pytest.mark.parametrize("G", [128, 64])
def test_knorm_full(orc, dev, G):
    run_knorm(orc, dev, W.knorm_paged(gamma_len=G))


@pytest.mark.parametrize("interleaved", [True, False])
def test_gqa_largest_head(orc, dev, interleaved):
    """head_size 512 (the largest supported) with 28 + 4 heads: 1024 rotation
    items per token, the limit of the mrope kernel's one-thread-per-item CTA."""
    for mode, sec in ((None, None), ("ids", None), ("mrope", (64, 96, 96))):
        w = W.gqa_workload("big", 450, [3, 0, 9, 1, 20], [0, 5, 40, 31, 7], 28, 4, 512,
                           page_size=16, freqs_rows=128, base=10000.0, interleaved=interleaved,
                           position_mode=mode, mrope_section=sec)
        run_gqa(orc, dev, w)


@pytest.mark.parametrize("G,S", [(100, 128), (8, 8), (24, 32), (256, 256), (512, 512),
                                 (1000, 1024), (2048, 2048)])
def test_knorm_widths(orc, dev, G, S):
    w = W.knorm_workload("w", 600 + G, [2, 0, 30, 1], [5, 0, 13, 61], 3, S, page_size=8,
                         gamma_len=G, spare_pages=2)
    run_knorm(orc, dev, w)


def test_knorm_variants(orc, dev):
    w = W.knorm_workload("v", 611, [2, 9, 1], [5, 0, 13], 4, 64, page_size=16, gamma_len=64,
                         weight_offset=0.5, multiply_before_cast=False)
    run_knorm(orc, dev, w)
    w = W.knorm_workload("v", 612, [2, 9, 1], [5, 0, 13], 4, 64, page_size=16, gamma_len=256)
    run_knorm(orc, dev, w, per_head_norm=False)
    # the widest whole-row norm: 4 heads x 512 = 2048 columns
    w = W.knorm_workload("v", 613, [2, 9, 1], [5, 0, 13], 4, 512, page_size=16, gamma_len=2048)
    run_knorm(orc, dev, w, per_head_norm=False)


def test_knorm_error_flags(orc, dev):
    w = W.knorm_workload("f", 613, [2, 3], [5, 20], 2, 32, page_size=8, gamma_len=32)
    w.cache.page_table[1, 2] = W.PAGE_UNMAPPED  # positions 16..23 of request 1
    d = run_knorm(orc, dev, w)
    assert d.flags() == 1


@pytest.mark.parametrize("G", [128, 64])
def test_knorm_full_with_bad_pages(orc, dev, G):
    """The benchmark batch with an unmapped page and a page id past the cache.
    With G = 128 the warps walk about 1.7 tiles each, so the kernel reads the
    page table from its shared-memory copy; with G = 64 (one tile per warp)
    from global memory."""
    w = W.knorm_paged(gamma_len=G)
    c = w.cache
    lens = np.diff(w.offsets.astype(np.int64))
    b1, b2 = [int(b) for b in np.flatnonzero(lens > 200)[:2]]
    p1 = int(c.cache_lengths[b1]) // c.page_size + 1
    p2 = int(c.cache_lengths[b2]) // c.page_size + 2
    c.page_table[b1, p1] = W.PAGE_UNMAPPED
    c.page_table[b2, p2] = c.num_pages + 5
    d = run_knorm(orc, dev, w)
    assert d.flags() == 1


# ------------------------------------------------------------ padded layouts, small batches

@pytest.mark.parametrize("kind", ["mla", "gqa", "gqa_mrope", "knorm", "gather", "gather_dynamic",
                                  "gather_dynamic_fp8"])
def test_padded_cache_layouts(orc, dev, kind):
    if kind.startswith("gather"):
        # padded rows: every latent row is copied from its own strided slot
        f8 = kind.endswith("fp8")
        w = W.mla_workload("p", 704, [3, 17, 1], [0, 40, 300], num_heads=1, page_size=16,
                           max_seq_len=512, cache_dtype=W.DTYPE_FP8_E4M3 if f8 else W.DTYPE_BF16,
                           num_layers=2, layer_idx=1, scale=1.0)
        w.cache = W.repad_cache(w.cache, 16, 32)
        run_gather(orc, dev, W.mla_gather(w, dynamic=kind != "gather"))
    elif kind == "mla":
        w = W.mla_workload("p", 701, [3, 17, 1], [0, 40, 300], num_heads=16, page_size=16,
                           max_seq_len=512, cache_dtype=W.DTYPE_BF16, num_layers=2, layer_idx=1)
        w.cache = W.repad_cache(w.cache, 64, 0)
        run_mla(orc, dev, w)
    elif kind.startswith("gqa"):
        mr = kind == "gqa_mrope"
        w = W.gqa_workload("p", 702, [3, 17, 1], [0, 40, 300], 8, 4, 128, page_size=16,
                           freqs_rows=512, base=500000.0, interleaved=not mr,
                           position_mode="mrope" if mr else None,
                           mrope_section=(16, 24, 24) if mr else None)
        w.cache = W.repad_cache(w.cache, 16, 32)  # kv heads not adjacent: per-head copies
        run_gqa(orc, dev, w)
    else:
        w = W.knorm_workload("p", 703, [3, 17, 1], [0, 40, 300], 4, 128, page_size=16,
                             gamma_len=96)
        w.cache = W.repad_cache(w.cache, 16, 32)
        run_knorm(orc, dev, w)


@pytest.mark.parametrize("new", [[1], [1, 1, 1], [5], [0, 2, 0, 0, 3], list(range(1, 40))])
def test_gqa_small_and_single_token_batches(orc, dev, new):
    prior = [7 * i for i in range(len(new))]
    for interleaved in (True, False):
        w = W.gqa_workload("t", 710 + len(new), new, prior, 32, 8, 128, page_size=64,
                           freqs_rows=1024, base=500000.0, interleaved=interleaved,
                           position_mode="ids")
        run_gqa(orc, dev, w)


def test_gqa_many_requests(orc, dev):
    rng = np.random.default_rng(9)
    B = 5000
    new = rng.integers(0, 3, B)
    prior = rng.integers(0, 500, B)
    w = W.gqa_workload("m", 720, new, prior, 4, 2, 64, page_size=8, freqs_rows=1024,
                       base=10000.0, interleaved=False, position_mode="mrope",
                       mrope_section=(6, 13, 13))
    run_gqa(orc, dev, w)


# ------------------------------------------------------------ MLA streaming (large batch) path

@pytest.mark.parametrize("H", [0, 1, 3, 5, 128])
@pytest.mark.parametrize("dtype", [W.DTYPE_FP8_E4M3, W.DTYPE_BF16])
def test_mla_stream_path_shapes(orc, dev, H, dtype):
    rng = np.random.default_rng(800 + H)
    new = rng.integers(500, 4000, 9)
    new[2] = 0
    new[5] = 1
    prior = rng.integers(0, 3000, 9)
    w = W.mla_workload("st", 801 + H, new, prior, num_heads=H, page_size=64,
                       max_seq_len=8192, cache_dtype=dtype, num_layers=2, layer_idx=1)
    run_mla(orc, dev, w)


def test_mla_stream_path_flags(orc, dev):
    rng = np.random.default_rng(811)
    new = rng.integers(2000, 4000, 6)
    prior = np.array([0, 100, 7000, 50, 6000, 10])
    w = W.mla_workload("sf", 812, new, prior, num_heads=16, page_size=64, max_seq_len=12288,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    w.freqs = w.freqs[:8192].copy()  # requests 2 and 4 run past the table
    w.cache.page_table[1, 3] = W.PAGE_UNMAPPED
    d, _, _ = run_mla(orc, dev, w)
    assert d.flags() == 3


# ------------------------------------------------------------ maximum request count

def test_max_batches_all_entry_points(orc, dev):
    """num_batches = 8192 (the documented maximum): the staged ragged tables
    take 64 KiB of shared memory in every kernel."""
    rng = np.random.default_rng(901)
    B = 8192
    new = rng.integers(0, 3, B)
    prior = rng.integers(0, 100, B)
    w = W.mla_workload("mb", 902, new, prior, num_heads=4, page_size=32, max_seq_len=128,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    assert w.B == B
    run_mla(orc, dev, w)
    g = W.gqa_workload("mb", 903, new, prior, 4, 2, 64, page_size=32, freqs_rows=128,
                       base=10000.0, interleaved=True, position_mode="ids")
    run_gqa(orc, dev, g)
    k = W.knorm_workload("mb", 904, new, prior, 2, 64, page_size=32, gamma_len=64)
    run_knorm(orc, dev, k)
    w2 = W.mla_workload("mb", 905, new, prior, num_heads=2, page_size=32, max_seq_len=128,
                        cache_dtype=W.DTYPE_BF16)
    run_mla(orc, dev, W.mla_inplace(w2))
    run_gather(orc, dev, W.mla_gather(w2, out_dtype=W.DTYPE_FP8_E4M3))


@pytest.mark.parametrize("name", ["knorm128_cast_first", "knorm_whole_row"])
def test_knorm_variant_configs_full(orc, dev, name):
    w = W.REGISTRY[name][0](2)
    run_knorm(orc, dev, w, per_head_norm=w.per_head_norm)



# ------------------------------------------------------------ FP8 q output, in-place variant

@pytest.mark.parametrize("build", ["tiny", "decode", "prefill"])
def test_mla_fp8_q_output(orc, dev, build):
    import dataclasses

    w = {"tiny": lambda: W.mla_tiny(W.DTYPE_FP8_E4M3), "decode": lambda: W.mla_decode(),
         "prefill": lambda: W.mla_prefill(W.DTYPE_FP8_E4M3)}[build]()
    run_mla(orc, dev, dataclasses.replace(w, q_out_dtype=W.DTYPE_FP8_E4M3))


def test_mla_inplace_fp8_q_output(orc, dev):
    import dataclasses

    w = W.mla_inplace(W.mla_decode(W.DTYPE_FP8_E4M3))
    run_mla(orc, dev, dataclasses.replace(w, q_out_dtype=W.DTYPE_FP8_E4M3))


@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
@pytest.mark.parametrize("build", ["tiny", "decode", "prefill", "odd"])
def test_mla_inplace(orc, dev, dtype, build):
    if build == "tiny":
        w = W.mla_tiny(dtype)
    elif build == "decode":
        w = W.mla_decode(dtype)
    elif build == "prefill":
        w = W.mla_prefill(dtype)
    else:  # stream path, odd head counts, empty requests, a second layer, scale 2
        rng = np.random.default_rng(820)
        new = rng.integers(300, 3000, 7)
        new[3] = 0
        w = W.mla_workload("ip", 821, new, rng.integers(0, 2000, 7), num_heads=3, page_size=64,
                           max_seq_len=8192, cache_dtype=dtype, num_layers=2, layer_idx=1,
                           scale=2.0)
    run_mla(orc, dev, W.mla_inplace(w))


def test_mla_inplace_flags(orc, dev):
    w = W.mla_workload("pf", 91, [2, 5], [0, 60], num_heads=2, page_size=16, max_seq_len=80,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    w.freqs = w.freqs[:64].copy()
    w = W.mla_inplace(w)
    w.cache.page_table[0, 0] = W.PAGE_UNMAPPED
    d, _, _ = run_mla(orc, dev, w)
    assert d.flags() == 3


# ------------------------------------------------------------ paged -> contiguous gather

def run_gather(orc, dev, g, launch=None):
    import torch

    d = dev.DeviceGather(g)
    (launch or _launch)(d)
    torch.cuda.synchronize()
    if g.dynamic:
        ref, ref_scales, f_ref = orc.mla_gather_latent_dynamic(
            g.cache, g.layer_idx, g.ctx_offsets, out=d.out_init.copy(),
            scales=np.zeros(g.rows, np.float32))
        assert d.guards_intact()
        assert d.flags() == f_ref
        assert np.array_equal(d.scales.host(), ref_scales)
        assert np.array_equal(d.out.host(), ref)
        assert np.array_equal(d.cache.host(), g.cache.data)
        return d
    ref, f_ref = orc.mla_gather_latent(g.cache, g.layer_idx, g.ctx_offsets, g.out_dtype,
                                       g.out_scale, out=d.out_init.copy())
    assert d.guards_intact()
    assert d.flags() == f_ref
    got = d.out.host()
    if g.out_dtype == W.DTYPE_BF16:
        assert np.array_equal(got, ref)  # a copy or an exact E4M3 -> bf16 widening
    else:
        compare_e4m3(got, ref)
    assert np.array_equal(d.cache.host(), g.cache.data)  # the cache is only read
    return d


@pytest.mark.parametrize("src", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
@pytest.mark.parametrize("dst", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
def test_gather_small(orc, dev, src, dst):
    w = W.mla_workload("g", 830, [3, 0, 17, 1, 40], [5, 9, 100, 31, 0], num_heads=1,
                       page_size=16, max_seq_len=256, cache_dtype=src, num_layers=2, layer_idx=1,
                       scale=0.5)
    run_gather(orc, dev, W.mla_gather(w, out_dtype=dst, out_scale=2.0))


@pytest.mark.parametrize("dst", [W.DTYPE_FP8_E4M3, W.DTYPE_BF16])
def test_gather_prefill_full(orc, dev, dst):
    run_gather(orc, dev, W.mla_gather(W.mla_prefill(W.DTYPE_BF16), out_dtype=dst))


@pytest.mark.parametrize("src,scale", [(W.DTYPE_BF16, 1.0), (W.DTYPE_FP8_E4M3, 1.0),
                                       (W.DTYPE_FP8_E4M3, 0.625)])
def test_gather_dynamic_small(orc, dev, src, scale):
    """Codes and scales bit for bit: bf16 values and FP8 at scale 1 take the
    reciprocal-and-FMA division, FP8 at another scale the IEEE divide."""
    w = W.mla_workload("g", 860, [3, 0, 17, 1, 40, 70], [5, 9, 100, 31, 0, 200], num_heads=1,
                       page_size=16, max_seq_len=512, cache_dtype=src, num_layers=2,
                       layer_idx=1, scale=scale)
    g = W.mla_gather(w, dynamic=True)
    run_gather(orc, dev, g)


def test_gather_dynamic_outliers_and_zero_rows(orc, dev):
    """Rows with x1000 outliers (tiny quotients elsewhere in the row) and an
    all-zero row (scale 1)."""
    w = W.mla_workload("g", 861, [30, 50], [10, 0], num_heads=1, page_size=16, max_seq_len=128,
                       cache_dtype=W.DTYPE_BF16)
    g = W.mla_gather(w, dynamic=True)
    v = g.cache.view6()
    rng = np.random.default_rng(862)
    for b in range(2):
        for p in range(int(g.ctx_offsets[b + 1] - g.ctx_offsets[b])):
            page = int(g.cache.page_table[b, p // 16])
            row = v[page, 0, g.layer_idx, p % 16, 0]
            if p == 3:
                row[:] = 0
            elif p % 4 == 1:
                big = np.array([1000.0 * (1 + rng.random())], np.float32)
                row[rng.integers(0, 576)] = W.bf16_bits(big)[0]
    run_gather(orc, dev, g)


@pytest.mark.parametrize("cache_dtype", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
def test_gather_dynamic_nan_values(orc, dev, cache_dtype):
    """NaN values in cached rows: the row maximum ignores them (as the
    reference maximum does), so the scales and every code of a non-NaN value
    match the reference bit for bit; a NaN value gives a NaN code (E4M3
    S.1111.111).  Some rows hold one NaN, one holds NaNs only, and the NaN
    sits in a lane's first piece, second piece or the 64-wide tail."""
    import torch

    w = W.mla_workload("gn", 871, [40, 30], [5, 0], num_heads=1, page_size=16,
                       max_seq_len=128, cache_dtype=cache_dtype)
    g = W.mla_gather(w, dynamic=True)
    v = g.cache.view6()
    nan_code = 0x7FC1 if cache_dtype == W.DTYPE_BF16 else 0x7F
    rng = np.random.default_rng(872)
    for b in range(2):
        for p in range(int(g.ctx_offsets[b + 1] - g.ctx_offsets[b])):
            page = int(g.cache.page_table[b, p // 16])
            row = v[page, 0, g.layer_idx, p % 16, 0]
            if p == 7:
                row[:] = nan_code
            elif p % 3 == 1:
                col = [3, 300, 520, int(rng.integers(0, 576))][p % 4]
                row[col] = nan_code | (0x8000 if cache_dtype == W.DTYPE_BF16 and p % 2 else 0)
    d = dev.DeviceGather(g)
    d.run()
    torch.cuda.synchronize()
    ref, ref_scales, f_ref = orc.mla_gather_latent_dynamic(
        g.cache, g.layer_idx, g.ctx_offsets, out=d.out_init.copy(),
        scales=np.zeros(g.rows, np.float32))
    assert d.guards_intact() and d.flags() == f_ref
    assert np.array_equal(d.scales.host(), ref_scales)
    got = d.out.host()
    src = np.stack([v[int(g.cache.page_table[b, p // 16]), 0, g.layer_idx, p % 16, 0]
                    for b in range(2) for p in range(int(g.ctx_offsets[b + 1] - g.ctx_offsets[b]))])
    if cache_dtype == W.DTYPE_BF16:
        is_nan = (src & 0x7FFF) > 0x7F80
    else:
        is_nan = (src & 0x7F) == 0x7F
    assert is_nan.any()
    assert np.array_equal(got[~is_nan], ref[~is_nan])
    assert np.all((got[is_nan] & 0x7F) == 0x7F)


def test_gather_dynamic_every_bf16_maximum(orc, dev):
    """Row r's largest magnitude is the bf16 pattern min(r, 0x7F80), from 0 and
    the subnormals through every binade to infinity, at column r % 576 with
    either sign; the other values are random patterns below it.  Scales
    (amax / 448) and codes bit for bit, so every row maximum takes the
    scale path the kernel gives it: the refined division by 448 in the normal
    range, the IEEE divide at both ends, and the IEEE divide of the values
    where the scale leaves the refined range."""
    n = 0x7F80 + 4
    w = W.mla_workload("gm", 880, [1, 1, 1, 1], [8200, 8200, 8200, n - 4 * 8201 + 8200],
                       num_heads=1, page_size=64, max_seq_len=8256, cache_dtype=W.DTYPE_BF16)
    g = W.mla_gather(w, dynamic=True)
    assert int(g.ctx_offsets[-1]) == n
    rng = np.random.default_rng(881)
    top = np.minimum(np.arange(n), 0x7F80).astype(np.int64)
    rows = (rng.random((n, 576)) * (top[:, None] + 1)).astype(np.int64)
    rows = np.minimum(rows, top[:, None])
    rows[np.arange(n), np.arange(n) % 576] = top
    rows |= rng.integers(0, 2, size=rows.shape) << 15
    rows = rows.astype(np.uint16)
    v = g.cache.view6()
    P = g.cache.page_size
    for b in range(4):
        lo, hi = int(g.ctx_offsets[b]), int(g.ctx_offsets[b + 1])
        p = np.arange(hi - lo)
        v[g.cache.page_table[b, p // P].astype(np.int64), 0, g.layer_idx, p % P, 0] = rows[lo:hi]
    import torch

    d = dev.DeviceGather(g)
    d.run()
    torch.cuda.synchronize()
    ref, ref_scales, f_ref = orc.mla_gather_latent_dynamic(
        g.cache, g.layer_idx, g.ctx_offsets, out=d.out_init.copy(),
        scales=np.zeros(g.rows, np.float32))
    assert d.guards_intact() and d.flags() == f_ref
    assert np.array_equal(d.scales.host(), ref_scales)
    got = d.out.host()
    # An infinite value in a row whose scale is infinite gives inf / inf, a NaN
    # whose sign IEEE 754 leaves open (the host's division picks one by
    # platform): NaN codes compare up to the sign, every other code exactly.
    is_nan = (ref & 0x7F) == 0x7F
    assert is_nan.sum() == np.count_nonzero((rows & 0x7FFF) == 0x7F80)
    assert np.array_equal(got[~is_nan], ref[~is_nan])
    assert np.all((got[is_nan] & 0x7F) == 0x7F)


@pytest.mark.parametrize("dynamic", [False, True])
def test_gather_most_requests(orc, dev, dynamic):
    """KVW_MAX_BATCHES requests of 0-5 context rows each: the staged offsets
    take 32 KiB of shared memory beside the stages, and the steps of a warp
    straddle many requests."""
    n = 8192
    rng = np.random.default_rng(890)
    prior = rng.integers(0, 5, size=n)
    new = (rng.random(n) < 0.5).astype(np.int64)
    w = W.mla_workload("gb", 891, new, prior, num_heads=1, page_size=4, max_seq_len=8,
                       cache_dtype=W.DTYPE_BF16)
    g = W.mla_gather(w, dynamic=dynamic)
    assert g.ctx_offsets.shape[0] - 1 == n and g.rows > 16000
    run_gather(orc, dev, g)


@pytest.mark.parametrize("scale", [1.0, 0.75])
def test_gather_dynamic_prefill_size_fp8_cache(orc, dev, scale):
    """Prefill-size contexts (16 requests of 512-8192 rows) from an E4M3 cache:
    at cache scale 1 the values are bf16 numbers and divide through the
    refined quotient, at 0.75 through the IEEE divide; codes and scales bit
    for bit."""
    new = np.random.default_rng(1407).integers(512, 8192, size=16, endpoint=True)
    w = W.mla_workload("gpf", 1408, new, np.zeros(16, np.int64), num_heads=1, page_size=128,
                       max_seq_len=16384, cache_dtype=W.DTYPE_FP8_E4M3, scale=scale)
    g = W.mla_gather(w, dynamic=True)
    assert g.rows > 40000
    run_gather(orc, dev, g)


def test_gather_dynamic_prefill_full(orc, dev):
    run_gather(orc, dev, W.REGISTRY["mla_gather_prefill_dynamic"][0](2))


def test_gather_dynamic_flags(orc, dev):
    w = W.mla_workload("g", 863, [3, 5], [0, 7], num_heads=1, page_size=16, max_seq_len=64,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    g = W.mla_gather(w, dynamic=True)
    g.cache.page_table[1, 0] = W.PAGE_UNMAPPED
    assert run_gather(orc, dev, g).flags() == 1


def test_gather_decode_contexts(orc, dev):
    run_gather(orc, dev, W.mla_gather(W.mla_decode(W.DTYPE_FP8_E4M3), out_dtype=W.DTYPE_BF16))


def test_gather_flags(orc, dev):
    w = W.mla_workload("g", 831, [3, 5], [0, 7], num_heads=1, page_size=16, max_seq_len=64,
                       cache_dtype=W.DTYPE_BF16)
    g = W.mla_gather(w)
    g.cache.page_table[1, 0] = W.PAGE_UNMAPPED
    assert run_gather(orc, dev, g).flags() == 1
    g = W.mla_gather(W.mla_workload("g", 832, [3, 5], [0, 7], num_heads=1, page_size=16,
                                    max_seq_len=64, cache_dtype=W.DTYPE_BF16))
    g.ctx_offsets = g.ctx_offsets.copy()
    g.ctx_offsets[1] = g.ctx_offsets[2] + 1  # decreasing
    assert run_gather(orc, dev, g).flags() == 4


# ------------------------------------------------------------ FP8 codecs

def test_convert_all_bf16_patterns_and_random(orc, dev):
    import torch

    from gqa_kv_cache_mla_gb300 import kvw

    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = (h.astype(np.uint32) << 16).view(np.float32)
    h = h[np.isfinite(v)]
    h = h[: h.size // 8 * 8]
    rng = np.random.default_rng(840)
    x = np.concatenate([h, W.normal_bf16(rng, (1 << 20,), std=3.0)])
    for scale in (1.0, 0.37):
        d = dev.Guarded(x, "cuda")
        out = dev.Guarded(np.zeros(x.size, np.uint8), "cuda")
        kvw.kvw_convert_bf16_to_fp8_e4m3(out.tensor, d.tensor, scale)
        torch.cuda.synchronize()
        assert out.guards_intact() and d.guards_intact()
        assert np.array_equal(out.host(), orc.convert_bf16_to_e4m3(x, scale))


@pytest.mark.parametrize("rows,cols", [(1, 8), (37, 576), (4096, 2048)])
def test_quantize_rows(orc, dev, rows, cols):
    import torch

    from gqa_kv_cache_mla_gb300 import kvw

    rng = np.random.default_rng(841 + rows)
    x = W.normal_bf16(rng, (rows, cols), outlier_frac=0.01)
    x[0, :] = 0  # an all-zero row: scale 1
    d = dev.Guarded(x, "cuda")
    out = dev.Guarded(np.zeros(x.shape, np.uint8), "cuda")
    sc = dev.Guarded(np.zeros(rows, np.float32), "cuda")
    kvw.kvw_quantize_fp8_rows(out.tensor, sc.tensor, d.tensor)
    torch.cuda.synchronize()
    assert out.guards_intact() and sc.guards_intact()
    codes, scales = orc.quantize_rows_e4m3(x)
    assert np.array_equal(sc.host(), scales)
    assert np.array_equal(out.host(), codes)


def quant_rows_mantissa_sweep(shift):
    """Rows for the per-row quantiser that meet every scale mantissa it can see
    with every bf16 value whose quotient can give a non-zero code.

    Up to a power of two, the row maximum a is one of 128 bf16 values in
    [1, 2), so scale = RN(a / 448) takes 128 mantissas.  For each a, the row
    group holds a itself and every bf16 x of either sign with
    2^-23 <= |x| <= a (quotients down to about 2^-14), plus zeros of both
    signs and a few subnormals; the whole group is then shifted by 2^shift
    (exponent field + shift) to reach other scale binades."""
    groups = []
    exps = np.arange(127 - 23, 128, dtype=np.uint16)
    allx = ((exps[:, None] << 7) | np.arange(128, dtype=np.uint16)[None, :]).reshape(-1)
    for ma in range(128):
        a = np.uint16(0x3F80 | ma)
        xs = allx[allx <= a]
        vals = np.concatenate([xs, xs | 0x8000]).astype(np.uint16)
        if shift:
            vals = (vals.astype(np.int32) + (shift << 7)).astype(np.uint16)
        a_s = np.uint16(int(a) + (shift << 7))
        extra = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x807F], np.uint16)
        vals = np.concatenate([vals, extra])
        per_row = 2047
        n_rows = -(-vals.size // per_row)
        block = np.zeros((n_rows, 2048), np.uint16)
        block[:, 0] = a_s
        flat = np.zeros(n_rows * per_row, np.uint16)
        flat[: vals.size] = vals
        block[:, 1:] = flat.reshape(n_rows, per_row)
        groups.append(block)
    return np.concatenate(groups)


@pytest.mark.parametrize("shift", [0, 40, -40, -80, 100])
def test_quantize_rows_every_scale_mantissa(orc, dev, shift):
    """Bit-exact codes and scales on the mantissa sweep: shifts 0 and +-40 use
    the reciprocal-and-FMA division, -80 and +100 (scales outside [2^-60,
    2^60]) the IEEE divide."""
    import torch

    from gqa_kv_cache_mla_gb300 import kvw

    x = quant_rows_mantissa_sweep(shift)
    d = dev.Guarded(x, "cuda")
    out = dev.Guarded(np.zeros(x.shape, np.uint8), "cuda")
    sc = dev.Guarded(np.zeros(x.shape[0], np.float32), "cuda")
    kvw.kvw_quantize_fp8_rows(out.tensor, sc.tensor, d.tensor)
    torch.cuda.synchronize()
    codes, scales = orc.quantize_rows_e4m3(x)
    assert np.array_equal(sc.host(), scales)
    got = out.host()
    bad = np.flatnonzero(got != codes)
    assert bad.size == 0, (bad.size, x.reshape(-1)[bad[:5]], got.reshape(-1)[bad[:5]],
                           codes.reshape(-1)[bad[:5]])


@pytest.mark.parametrize("rows,cols,in_stride,out_stride", [
    (24, 4096, 4096, 4096),    # longer than 2048: the two-pass kernel
    (33, 3000, 3008, 3000),    # ragged last vector group, padded input rows
    (40, 576, 640, 600),       # register kernel with strided rows on both sides
])
def test_quantize_rows_long_and_strided(orc, dev, rows, cols, in_stride, out_stride):
    import torch

    from gqa_kv_cache_mla_gb300 import kvw

    rng = np.random.default_rng(850 + cols)
    x = W.normal_bf16(rng, (rows, in_stride), outlier_frac=0.02)
    d = dev.Guarded(x, "cuda")
    out0 = np.full((rows, out_stride), 0x5A, np.uint8)
    out = dev.Guarded(out0, "cuda")
    sc = dev.Guarded(np.zeros(rows, np.float32), "cuda")
    kvw.kvw_quantize_fp8_rows(out.tensor, sc.tensor, d.tensor, rows=rows, cols=cols,
                              in_row_stride=in_stride, out_row_stride=out_stride)
    torch.cuda.synchronize()
    assert out.guards_intact() and sc.guards_intact()
    codes, scales = orc.quantize_rows_e4m3(np.ascontiguousarray(x[:, :cols]))
    got = out.host()
    assert np.array_equal(sc.host(), scales)
    assert np.array_equal(got[:, :cols], codes)
    assert np.array_equal(got[:, cols:], out0[:, cols:])  # the row padding is not written


def test_convert_benchmark_shape(orc, dev):
    """The 2^26-value launch the benchmark times, every code compared."""
    import torch

    w = W.fp8_convert()
    d = dev.DeviceConvert(w)
    d.run()
    torch.cuda.synchronize()
    assert d.guards_intact()
    assert np.array_equal(d.out.host(), orc.convert_bf16_to_e4m3(w.x, w.scale))


def test_quantize_rows_benchmark_shape(orc, dev):
    import torch

    w = W.fp8_quant_rows()
    d = dev.DeviceConvert(w)
    d.run()
    torch.cuda.synchronize()
    codes, scales = orc.quantize_rows_e4m3(w.x)
    assert np.array_equal(d.scales.host(), scales) and np.array_equal(d.out.host(), codes)
