"""Pins for the oracle's FP8 details and the in-place / gather MLA steps.

* FP8 q_rope output: the rotation decoded from E4M3 is within one E4M3
  rounding of the float64 complex rotation; at position 0 it equals the
  library cast of the input.
* convert_bf16_to_fp8_e4m3fn: the library cast (scale 1); scale s on x equals
  scale 1 on x / s for powers of two.
* dynamic per-row FP8: closed form -- the row maximum maps to 448, every
  code equals the library cast of x / scale.
* in-place MLA: placing the latent rows in the cache and running the
  in-place variant equals the fused write (bf16 cache, and FP8 cache with
  scale 1 since every E4M3 value is a bf16 value).
* paged -> contiguous gather: brute force over the slot formula; bf16 ->
  bf16 is a copy, bf16 -> FP8 the library cast of value / scale, FP8 -> bf16
  the decoded value times the scale.
"""
import numpy as np
import pytest
import torch

from gqa_kv_cache_mla_gb300 import workloads as W
from helpers import bf16_to_f32, expected_slots


def _torch_e4m3(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def _theta(dim, base):
    return base ** (-2.0 * np.arange(dim // 2, dtype=np.float64) / dim)


def test_fp8_q_output_vs_complex_fp64(orc):
    w = W.mla_tiny()
    q8, _, flags = orc.mla_rope_rmsnorm_quant(w, out_dtype=1)
    assert flags == 0 and q8.dtype == np.uint8
    c = w.cache
    theta = _theta(64, 10000.0)
    x = bf16_to_f32(w.q_rope).astype(np.float64)
    y = orc.e4m3_decode(q8).astype(np.float64)
    for t, _, _, pos in expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size):
        z = (x[t, :, 0::2] + 1j * x[t, :, 1::2]) * np.exp(1j * pos * theta)
        for got, want in ((y[t, :, 0::2], z.real), (y[t, :, 1::2], z.imag)):
            assert np.all(np.abs(got - want) <= np.abs(want) * 2.0**-4 + 2.0**-10 + 1e-6)


def test_fp8_q_output_position_zero_is_library_cast(orc):
    w = W.mla_workload("z", 31, [1, 1, 1], [0, 0, 0], num_heads=3, page_size=16,
                       max_seq_len=32, cache_dtype=W.DTYPE_BF16)
    q8, _, _ = orc.mla_rope_rmsnorm_quant(w, out_dtype=1)
    assert np.array_equal(q8, _torch_e4m3(bf16_to_f32(w.q_rope)))


def test_convert_matches_library_cast(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bf16_to_f32(h)
    ok = np.isfinite(v) & (np.abs(v) <= 464)
    assert np.array_equal(orc.convert_bf16_to_e4m3(h[ok]), _torch_e4m3(v[ok]))
    big = h[np.isfinite(v) & (np.abs(v) > 464)]
    codes = orc.convert_bf16_to_e4m3(big)
    assert np.all((codes & 0x7F) == 0x7E)  # saturates to +-448


@pytest.mark.parametrize("k", [1, -2, 4])
def test_convert_scale_is_a_division(orc, k):
    rng = np.random.default_rng(5)
    x = W.bf16_bits(rng.standard_normal(4096).astype(np.float32) * 3)
    s = 2.0**k
    a = orc.convert_bf16_to_e4m3(x, scale=s)
    b = orc.convert_bf16_to_e4m3(W.bf16_bits(bf16_to_f32(x) / np.float32(s)))
    assert np.array_equal(a, b)


def test_dynamic_row_quantisation_closed_form(orc):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((64, 576)).astype(np.float32) * rng.uniform(0.01, 100, (64, 1))
    x[3] = 0.0
    xb = W.bf16_bits(x)
    codes, sc = orc.quantize_rows_e4m3(xb)
    xv = bf16_to_f32(xb)
    amax = np.abs(xv).max(axis=1)
    assert sc[3] == 1.0 and not codes[3].any()
    nz = amax > 0
    assert np.array_equal(sc[nz], (amax[nz] / np.float32(448.0)).astype(np.float32))
    for r in np.flatnonzero(nz):
        want = _torch_e4m3(xv[r] / sc[r])
        assert np.array_equal(codes[r], want)
        assert np.max(np.abs(orc.e4m3_decode(codes[r]))) == 448.0


@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_FP8_E4M3])
def test_inplace_equals_fused_write(orc, dtype):
    w = W.mla_workload("ip", 171, [3, 5, 0, 9], [0, 7, 3, 40], num_heads=4, page_size=16,
                       max_seq_len=128, cache_dtype=dtype, num_layers=2, layer_idx=1,
                       spare_pages=2)
    if dtype == W.DTYPE_FP8_E4M3:  # the fused input must be the value the cache holds
        w.kv_in = W.bf16_bits(orc.e4m3_decode(_torch_e4m3(bf16_to_f32(w.kv_in))))
    q_f, c_f, f1 = orc.mla_rope_rmsnorm_quant(w)
    W.place_latent_rows(w)
    q_i, c_i, f2 = orc.mla_rope_rmsnorm_inplace(w)
    assert f1 == f2 == 0
    assert np.array_equal(q_f, q_i)
    assert np.array_equal(c_f, c_i)


def _gather_case(dtype, scale=1.0):
    w = W.mla_workload("g", 181, [3, 5, 0, 9], [0, 7, 3, 40], num_heads=1, page_size=16,
                       max_seq_len=128, cache_dtype=dtype, scale=scale, num_layers=2,
                       layer_idx=1)
    ctx = W.context_offsets(w.cache, w.offsets)
    # a cache holds normalised latent rows: N(0,1) values in every context slot
    rng = np.random.default_rng(182)
    c = w.cache
    v = c.view6()
    for b in range(len(ctx) - 1):
        for p in range(int(ctx[b + 1]) - int(ctx[b])):
            x = rng.standard_normal(576).astype(np.float32)
            page = int(c.page_table[b, p // c.page_size])
            v[page, 0, w.layer_idx, p % c.page_size, 0] = (
                W.bf16_bits(x) if dtype == W.DTYPE_BF16 else W.e4m3_bits(x / np.float32(scale)))
    return w, ctx


def _expected_rows(w, ctx):
    c = w.cache
    v = c.view6()
    out = {}
    for b in range(len(ctx) - 1):
        for p in range(int(ctx[b + 1]) - int(ctx[b])):
            page = int(c.page_table[b, p // c.page_size])
            out[int(ctx[b]) + p] = v[page, 0, w.layer_idx, p % c.page_size, 0]
    return out


@pytest.mark.parametrize("src,dst", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gather_brute_force(orc, src, dst):
    w, ctx = _gather_case(src)
    out, flags = orc.mla_gather_latent(w.cache, w.layer_idx, ctx, out_dtype=dst,
                                       out_scale=2.0 if (src, dst) == (0, 1) else 1.0)
    assert flags == 0
    rows = _expected_rows(w, ctx)
    assert len(rows) == out.shape[0] == int(ctx[-1])
    for r, raw in rows.items():
        if src == dst:
            assert np.array_equal(out[r], raw)
        elif src == 0:  # bf16 -> fp8 with scale 2
            assert np.array_equal(out[r], _torch_e4m3(bf16_to_f32(raw) / 2.0))
        else:  # fp8 -> bf16: decoded value (exact in bf16)
            assert np.array_equal(bf16_to_f32(out[r]), orc.e4m3_decode(raw))


def test_gather_flags(orc):
    w, ctx = _gather_case(0)
    w.cache.page_table[1, 0] = W.PAGE_UNMAPPED
    out, flags = orc.mla_gather_latent(w.cache, w.layer_idx, ctx)
    assert flags == orc.FLAG_PAGE
    assert not out[int(ctx[1]):int(ctx[2])].any()  # request 1 (one page, unmapped) is skipped
    bad = ctx.copy()
    bad[2] = bad[1] - 1
    _, flags = orc.mla_gather_latent(w.cache, w.layer_idx, bad)
    assert flags == orc.FLAG_OFFSETS


def test_gather_fp8_cache_scale(orc):
    """An FP8 cache is read as code value times the cache scale."""
    w, ctx = _gather_case(W.DTYPE_FP8_E4M3, scale=2.0)
    out, flags = orc.mla_gather_latent(w.cache, w.layer_idx, ctx, out_dtype=W.DTYPE_BF16)
    assert flags == 0
    for r, raw in _expected_rows(w, ctx).items():
        assert np.array_equal(bf16_to_f32(out[r]), orc.e4m3_decode(raw) * np.float32(2.0))


# ------------------------------------------------------------ gather with dynamic per-row FP8

def test_gather_dynamic_equals_gather_then_row_quantisation(orc):
    """bf16 cache: the fused copy + per-row dynamic FP8 equals the plain copy
    (bf16 out, an exact copy) followed by the per-row quantiser, codes and
    scales bit for bit."""
    w, ctx = _gather_case(W.DTYPE_BF16)
    rows, flags = orc.mla_gather_latent(w.cache, w.layer_idx, ctx, out_dtype=W.DTYPE_BF16)
    want_codes, want_scales = orc.quantize_rows_e4m3(rows)
    codes, scales, f2 = orc.mla_gather_latent_dynamic(w.cache, w.layer_idx, ctx)
    assert flags == f2 == 0
    assert np.array_equal(scales, want_scales)
    assert np.array_equal(codes, want_codes)


def test_gather_dynamic_closed_form_fp8_cache(orc):
    """FP8 cache with scale 0.75: each row's values are code x 0.75, its scale
    is max|value| / 448, its largest magnitude becomes +-448 and every code is
    torch's E4M3 cast of value / scale."""
    w, ctx = _gather_case(W.DTYPE_FP8_E4M3, scale=0.75)
    codes, scales, flags = orc.mla_gather_latent_dynamic(w.cache, w.layer_idx, ctx)
    assert flags == 0
    for r, raw in _expected_rows(w, ctx).items():
        v = orc.e4m3_decode(raw) * np.float32(0.75)
        amax = np.float32(np.abs(v).max())
        assert scales[r] == np.float32(amax / np.float32(448.0))
        assert np.array_equal(codes[r], _torch_e4m3(v / scales[r]))
        assert np.abs(orc.e4m3_decode(codes[r])).max() == 448.0


def test_gather_dynamic_flags_and_zero_rows(orc):
    w, ctx = _gather_case(W.DTYPE_BF16)
    c = w.cache
    v = c.view6()
    page = int(c.page_table[3, 0])
    v[page, 0, w.layer_idx, 0, 0, :] = 0  # request 3's first row: all zeros -> scale 1
    c.page_table[1, 0] = W.PAGE_UNMAPPED
    codes, scales, flags = orc.mla_gather_latent_dynamic(w.cache, w.layer_idx, ctx)
    assert flags == orc.FLAG_PAGE
    assert not codes[int(ctx[1]):int(ctx[2])].any() and not scales[int(ctx[1]):int(ctx[2])].any()
    r0 = int(ctx[3])
    assert scales[r0] == 1.0 and not codes[r0].any()
    bad = ctx.copy()
    bad[2] = bad[1] - 1
    codes, scales, flags = orc.mla_gather_latent_dynamic(w.cache, w.layer_idx, bad)
    assert flags == orc.FLAG_OFFSETS and not codes.any() and not scales.any()
