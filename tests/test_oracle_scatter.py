"""Brute-force pins for the oracle's ragged -> paged addressing.

The expected set of written cache rows is enumerated in the test by the slot
formula (token i of request b lands at position cache_lengths[b] + i, row
position % page_size of page page_table[b][position // page_size]); the
oracle must change bytes only inside that set and must leave every other
byte, including spare pages, other layers and V, as it was.  Also pinned:
error flags and composition identities.
"""
import numpy as np
import pytest

from gqa_kv_cache_mla_gb300 import workloads as W
from helpers import expected_slots


def _mask_rows(c, slots, layer, heads=None, cols=None):
    """Boolean mask over the cache (6-d) selecting K rows of the given slots."""
    m = np.zeros(c.view6().shape, dtype=bool)
    for _, page, row, _ in slots:
        if heads is None and cols is None:
            m[page, 0, layer, row] = True
        else:
            m[page, 0, layer, row, :, : (cols if cols is not None else c.head_size)] = True
    return m


@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
def test_mla_tiny_writes_exactly_new_rows(orc, dtype):
    w = W.mla_tiny(cache_dtype=dtype)
    c = w.cache
    assert c.num_pages == 8 and c.num_layers == 2 and w.layer_idx == 1
    slots = expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size)
    assert [s[3] for s in slots] == [0, 1, 2, 7, 8, 9, 10, 11]
    q_out0 = np.full(w.q_rope.shape, 0xABCD, np.uint16)
    q_out, cache, flags = orc.mla_rope_rmsnorm_quant(w, q_rope_out=q_out0.copy())
    assert flags == 0
    before = c.view6()
    after = cache.reshape(before.shape)
    m = _mask_rows(c, slots, w.layer_idx)
    assert np.array_equal(after[~m], before[~m])
    # every written row differs from its random prior contents somewhere
    for _, page, row, _ in slots:
        assert not np.array_equal(after[page, 0, w.layer_idx, row], before[page, 0, w.layer_idx, row])
    assert not np.any(q_out == 0xABCD)


def test_gqa_rotates_only_new_k_rows(orc):
    w = W.gqa_workload("g", 71, [3, 5, 0, 2], [0, 7, 4, 30], num_q_heads=4, num_kv_heads=2,
                       head_size=32, page_size=16, freqs_rows=64, base=10000.0,
                       interleaved=False, spare_pages=3)
    c = w.cache
    slots = expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size)
    out, cache, flags = orc.qk_rope_paged_ragged(w)
    assert flags == 0
    before = c.view6()
    after = cache.reshape(before.shape)
    m = _mask_rows(c, slots, w.layer_idx)
    assert np.array_equal(after[~m], before[~m])  # V, other layers, other slots, spares
    assert np.array_equal(after[:, 1], before[:, 1])
    changed = (after != before).any(axis=(4, 5))
    for _, page, row, pos in slots:  # position 0 rotates by angle 0: identity
        assert changed[page, 0, w.layer_idx, row] == (pos > 0)
    assert changed.sum() == sum(1 for s in slots if s[3] > 0)


def test_knorm_touches_only_leading_cols_of_new_rows(orc):
    G = 16
    w = W.knorm_workload("k", 81, [2, 0, 4, 1], [5, 0, 13, 31], num_kv_heads=2, head_size=32,
                         page_size=8, gamma_len=G, spare_pages=2)
    c = w.cache
    slots = expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size)
    cache, flags = orc.rms_norm_kv_cache_paged(w)
    assert flags == 0
    before = c.view6()
    after = cache.reshape(before.shape)
    m = _mask_rows(c, slots, w.layer_idx, heads=True, cols=G)
    assert np.array_equal(after[~m], before[~m])
    assert (after[m] != before[m]).mean() > 0.5


# ------------------------------------------------------------------ flags

def test_invalid_offsets_write_nothing(orc):
    for bad in ([1, 3, 8], [0, 5, 3, 8], [0, 3, 7]):
        w = W.mla_tiny()
        off = np.array(bad, np.uint32)
        w.offsets = off
        q0 = np.full(w.q_rope.shape, 0x1234, np.uint16)
        # T stays 8, so the last offset must be 8
        q_out, cache, flags = orc.mla_rope_rmsnorm_quant(w, q_rope_out=q0.copy(), T=8)
        if bad[-1] == 8 and bad[0] == 0 and all(a <= b for a, b in zip(bad, bad[1:])):
            continue
        assert flags == orc.FLAG_OFFSETS
        assert np.array_equal(q_out, q0)
        assert np.array_equal(cache, w.cache.data)


def test_position_past_table_skips_token(orc):
    # request 1 runs from position 60 to 64: position 64 is past a 64-row table
    w = W.mla_workload("p", 91, [2, 5], [0, 60], num_heads=2, page_size=16, max_seq_len=80,
                       cache_dtype=W.DTYPE_BF16)
    w.freqs = w.freqs[:64].copy()
    q0 = np.full(w.q_rope.shape, 0x1234, np.uint16)
    q_out, cache, flags = orc.mla_rope_rmsnorm_quant(w, q_rope_out=q0.copy())
    assert flags == orc.FLAG_POS
    # tokens 6 (position 64) is skipped entirely; the others are written
    assert np.array_equal(q_out[6], q0[6])
    assert not np.any(q_out[:6] == 0x1234)
    c = w.cache
    slots = expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size)
    before = c.view6()
    after = cache.reshape(before.shape)
    for t, page, row, pos in slots:
        same = np.array_equal(after[page, 0, 0, row], before[page, 0, 0, row])
        assert same == (pos >= 64)


def test_unmapped_page_skips_cache_row_only(orc):
    w = W.mla_tiny()
    c = w.cache
    # request 1 positions 7..11 all live in its page 0
    c.page_table[1, 0] = W.PAGE_UNMAPPED
    q_out, cache, flags = orc.mla_rope_rmsnorm_quant(w)
    assert flags == orc.FLAG_PAGE
    w2 = W.mla_tiny()
    q_ref, cache_ref, _ = orc.mla_rope_rmsnorm_quant(w2)
    assert np.array_equal(q_out, q_ref)  # q rows are written regardless of the page
    # cache: only request 0's rows changed
    before = c.view6()
    after = cache.reshape(before.shape)
    slots0 = [s for s in expected_slots(w2.offsets, w2.cache.cache_lengths,
                                        w2.cache.page_table, 16) if s[0] < 3]
    m = _mask_rows(c, slots0, w.layer_idx)
    assert np.array_equal(after[~m], before[~m])
    # a page id past num_pages is treated the same way
    w3 = W.mla_tiny()
    w3.cache.page_table[1, 0] = 8
    _, cache3, flags3 = orc.mla_rope_rmsnorm_quant(w3)
    assert flags3 == orc.FLAG_PAGE and np.array_equal(cache3, cache)


def test_gqa_flags(orc):
    w = W.gqa_workload("g", 72, [3, 5], [0, 7], num_q_heads=2, num_kv_heads=2, head_size=16,
                       page_size=16, freqs_rows=64, base=10000.0, interleaved=True,
                       position_mode="ids")
    w.position_ids[4] = 64  # past the table
    w.cache.page_table[0, 0] = W.PAGE_UNMAPPED
    out0 = np.full(w.q_proj.shape, 0x1111, np.uint16)
    out, cache, flags = orc.qk_rope_paged_ragged(w, output=out0.copy())
    assert flags == orc.FLAG_POS | orc.FLAG_PAGE
    assert np.array_equal(out[4], out0[4])
    assert not np.any(out[[0, 1, 2, 3, 5, 6, 7]] == 0x1111)


def test_empty_batch_is_a_no_op(orc):
    w = W.mla_workload("e", 93, [0, 0], [3, 0], num_heads=2, page_size=16, max_seq_len=32,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    assert w.T == 0
    q_out, cache, flags = orc.mla_rope_rmsnorm_quant(w)
    assert flags == 0 and np.array_equal(cache, w.cache.data)


# ------------------------------------------------------------ composition

def test_mla_without_q_heads_is_the_cache_write(orc):
    w4 = W.mla_workload("h", 101, [3, 5], [0, 7], num_heads=4, page_size=16, max_seq_len=64,
                        cache_dtype=W.DTYPE_FP8_E4M3)
    w0 = W.mla_workload("h", 101, [3, 5], [0, 7], num_heads=4, page_size=16, max_seq_len=64,
                        cache_dtype=W.DTYPE_FP8_E4M3)
    w0.q_rope = np.zeros((w0.T, 0, 64), np.uint16)
    _, c4, f4 = orc.mla_rope_rmsnorm_quant(w4)
    _, c0, f0 = orc.mla_rope_rmsnorm_quant(w0)
    assert f4 == f0 == 0 and np.array_equal(c4, c0)


def test_gqa_k_rotation_equals_q_rotation_of_a_copy(orc):
    w = W.gqa_workload("g", 73, [3, 5], [0, 7], num_q_heads=2, num_kv_heads=2, head_size=32,
                       page_size=16, freqs_rows=64, base=10000.0, interleaved=False,
                       position_mode="mrope", mrope_section=(4, 6, 6))
    c = w.cache
    slots = expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size)
    v = c.view6()
    k_rows = np.stack([v[page, 0, w.layer_idx, row] for _, page, row, _ in slots])
    w.q_proj = k_rows.copy()  # Hq = Hk, tokens in slot order
    out, cache, flags = orc.qk_rope_paged_ragged(w)
    assert flags == 0
    after = cache.reshape(v.shape)
    for i, (_, page, row, _) in enumerate(slots):
        assert np.array_equal(after[page, 0, w.layer_idx, row], out[i])


def test_gqa_output_may_alias_input(orc):
    w = W.gqa_workload("g", 74, [4, 2], [3, 0], num_q_heads=3, num_kv_heads=1, head_size=16,
                       page_size=16, freqs_rows=64, base=10000.0, interleaved=True)
    ref, _, _ = orc.qk_rope_paged_ragged(w)
    buf = w.q_proj.copy()
    w.q_proj = buf
    out, _, _ = orc.qk_rope_paged_ragged(w, output=buf)
    assert np.array_equal(buf, ref)


def test_fp8_scale_convention(orc):
    """stored = satfinite_rne(y / scale): doubling gamma and the rope part and
    using scale 2 gives the same codes as the unscaled case."""
    a = W.mla_workload("s", 111, [3, 5], [0, 7], num_heads=1, page_size=16, max_seq_len=64,
                       cache_dtype=W.DTYPE_FP8_E4M3)
    b = W.mla_workload("s", 111, [3, 5], [0, 7], num_heads=1, page_size=16, max_seq_len=64,
                       cache_dtype=W.DTYPE_FP8_E4M3, scale=2.0)
    from helpers import bf16_to_f32

    b.gamma = W.bf16_bits(bf16_to_f32(a.gamma) * 2)
    kv = bf16_to_f32(a.kv_in)
    kv[:, 512:] *= 2
    b.kv_in = W.bf16_bits(kv)
    _, ca, fa = orc.mla_rope_rmsnorm_quant(a)
    _, cb, fb = orc.mla_rope_rmsnorm_quant(b)
    assert fa == fb == 0
    assert np.array_equal(ca, cb)
    # and scale 1 vs scale 2 without the doubling do differ
    b2 = W.mla_workload("s", 111, [3, 5], [0, 7], num_heads=1, page_size=16, max_seq_len=64,
                        cache_dtype=W.DTYPE_FP8_E4M3, scale=2.0)
    _, cb2, _ = orc.mla_rope_rmsnorm_quant(b2)
    assert not np.array_equal(ca, cb2)


def test_openmp_threads_give_identical_results(orc):
    w = W.mla_workload("o", 121, [40, 1, 77, 9], [5, 300, 0, 1000], num_heads=8,
                       page_size=16, max_seq_len=2048, cache_dtype=W.DTYPE_FP8_E4M3)
    a = orc.mla_rope_rmsnorm_quant(w, nthreads=1)
    b = orc.mla_rope_rmsnorm_quant(w, nthreads=4)
    assert a[2] == b[2] == 0
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------ padded layouts

def test_layout_independence(orc):
    """The same logical cache in a padded layout (spare elements after every
    head and token row) gives the same logical result, and the spare
    elements are never touched."""
    from helpers import bf16_to_f32  # noqa: F401

    cases = [
        ("mla", W.mla_tiny(cache_dtype=W.DTYPE_FP8_E4M3), 0, 32),
        ("gqa", W.gqa_workload("p", 131, [3, 5, 1], [0, 7, 30], 4, 2, 32, page_size=16,
                               freqs_rows=64, base=10000.0, interleaved=False,
                               position_mode="mrope", mrope_section=(4, 6, 6)), 8, 16),
        ("knorm", W.knorm_workload("p", 132, [3, 5, 1], [0, 7, 30], 3, 32, page_size=8,
                                   gamma_len=24), 8, 24),
    ]
    for kind, w, head_pad, token_pad in cases:
        dense = w.cache
        padded = W.repad_cache(dense, head_pad, token_pad)
        run = {"mla": orc.mla_rope_rmsnorm_quant, "gqa": orc.qk_rope_paged_ragged,
               "knorm": orc.rms_norm_kv_cache_paged}[kind]
        out_d = run(w)
        w.cache = padded
        out_p = run(w)
        cache_d, cache_p = out_d[-2], out_p[-2]
        assert out_d[-1] == out_p[-1] == 0
        assert np.array_equal(dense.view6(cache_d), padded.view6(cache_p))
        if kind != "knorm":
            assert np.array_equal(out_d[0], out_p[0])
        # spare elements untouched
        n = padded.data.size
        used = np.zeros(n, dtype=bool)
        used[padded.view6(np.arange(n, dtype=np.int64)).reshape(-1)] = True
        assert np.array_equal(cache_p[~used], padded.data[~used])
