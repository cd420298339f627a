"""Pins for the oracle's rotary position embedding (RoPE) steps.

Closed forms: a rotation preserves each pair's length, the angle-0 rotation is
the identity, rotations compose additively.  Library special case: the
rotation of pair (x0, x1) by angle a equals the complex product
(x0 + i x1) * exp(i a), evaluated here in float64 by torch with angles taken
from theta_i = base^(-2i/D) directly (not from the table the oracle reads).
"""
import numpy as np
import pytest
import torch

from gqa_kv_cache_mla_gb300 import workloads as W
from helpers import bf16_to_f32


def _exact_rotation(x0, x1, ang):
    """(x0 + i x1) * exp(i ang) in complex128."""
    f = lambda a: torch.from_numpy(np.array(a, dtype=np.float64, copy=True))
    a = f(np.broadcast_to(ang, np.shape(x0)))
    r = torch.complex(f(x0), f(x1)) * torch.polar(torch.ones_like(a), a)
    return r.real.numpy(), r.imag.numpy()


def _theta(dim, base):
    return base ** (-2.0 * np.arange(dim // 2, dtype=np.float64) / dim)


def test_rope_pairs_vs_complex_fp64(orc):
    rng = np.random.default_rng(21)
    n = 100000
    x = rng.standard_normal(2 * n).astype(np.float32) * np.float32(3)
    ang = rng.uniform(-1000, 1000, n)
    cs = np.empty(2 * n, np.float32)
    cs[0::2] = np.cos(ang)
    cs[1::2] = np.sin(ang)
    y = orc.rope_pairs_f32(x, cs).astype(np.float64)
    e0, e1 = _exact_rotation(x[0::2], x[1::2], ang)
    bound = 8 * 2.0**-24 * (np.abs(x[0::2]) + np.abs(x[1::2])) + 1e-30
    assert np.all(np.abs(y[0::2] - e0) <= bound)
    assert np.all(np.abs(y[1::2] - e1) <= bound)


def test_rope_preserves_pair_norm(orc):
    rng = np.random.default_rng(22)
    n = 100000
    x = rng.standard_normal(2 * n).astype(np.float32)
    tab = W.rope_table(4096, 64, 10000.0)
    rows = rng.integers(0, 4096, n // 32)
    cs = tab[rows].reshape(-1)
    y = orc.rope_pairs_f32(x, cs).astype(np.float64)
    nx = x[0::2].astype(np.float64) ** 2 + x[1::2].astype(np.float64) ** 2
    ny = y[0::2] ** 2 + y[1::2] ** 2
    assert np.all(np.abs(np.sqrt(ny) - np.sqrt(nx)) <= 4 * 2.0**-24 * 2 * np.sqrt(nx) + 1e-30)


def test_rope_position_zero_is_identity(orc):
    tab = W.rope_table(1, 128, 500000.0)
    assert np.array_equal(tab[0, 0::2], np.ones(64, np.float32))
    assert np.array_equal(tab[0, 1::2], np.zeros(64, np.float32))
    rng = np.random.default_rng(23)
    x = rng.standard_normal(128 * 500).astype(np.float32)
    y = orc.rope_pairs_f32(x, np.tile(tab[0], 500))
    assert np.array_equal(y, x)


def test_rope_composes_additively(orc):
    rng = np.random.default_rng(24)
    tab = W.rope_table(8192, 128, 500000.0)
    x = rng.standard_normal(128 * 200).astype(np.float32)
    p1 = rng.integers(0, 4096, 200)
    p2 = rng.integers(0, 4096, 200)
    y12 = orc.rope_pairs_f32(orc.rope_pairs_f32(x, tab[p1].reshape(-1)), tab[p2].reshape(-1))
    y3 = orc.rope_pairs_f32(x, tab[p1 + p2].reshape(-1))
    assert np.max(np.abs(y12.astype(np.float64) - y3)) <= 64 * 2.0**-24 * np.max(np.abs(x)) * 2


# ---------------------------------------------------------- through the MLA entry

def _decode_cache_rows(w, cache):
    from helpers import expected_slots

    c = w.cache
    v = cache.reshape(c.num_pages, c.kv_dim, c.num_layers, c.page_size, c.num_heads,
                      c.head_size)
    rows = {}
    for t, page, row, pos in expected_slots(w.offsets, c.cache_lengths, c.page_table,
                                            c.page_size):
        rows[t] = (v[page, 0, w.layer_idx, row, 0, :].copy(), pos)
    return rows


def test_mla_q_and_k_rope_vs_complex_fp64(orc):
    w = W.mla_tiny()
    q_out, cache, flags = orc.mla_rope_rmsnorm_quant(w)
    assert flags == 0
    theta = _theta(64, 10000.0)
    rows = _decode_cache_rows(w, cache)
    x = bf16_to_f32(w.q_rope).astype(np.float64)
    y = bf16_to_f32(q_out).astype(np.float64)
    for t, (row, pos) in rows.items():
        ang = pos * theta
        e0, e1 = _exact_rotation(x[t, :, 0::2], x[t, :, 1::2], np.broadcast_to(ang, (w.H, 32)))
        tol0 = np.abs(e0) * 2.0**-8 + 1e-6 * (np.abs(x[t, :, 0::2]) + np.abs(x[t, :, 1::2]))
        tol1 = np.abs(e1) * 2.0**-8 + 1e-6 * (np.abs(x[t, :, 0::2]) + np.abs(x[t, :, 1::2]))
        assert np.all(np.abs(y[t, :, 0::2] - e0) <= tol0)
        assert np.all(np.abs(y[t, :, 1::2] - e1) <= tol1)
        kx = bf16_to_f32(w.kv_in[t, 512:]).astype(np.float64)
        ky = bf16_to_f32(row[512:]).astype(np.float64)
        k0, k1 = _exact_rotation(kx[0::2], kx[1::2], ang)
        assert np.all(np.abs(ky[0::2] - k0) <= np.abs(k0) * 2.0**-8 + 1e-6 * np.abs(kx).sum())
        assert np.all(np.abs(ky[1::2] - k1) <= np.abs(k1) * 2.0**-8 + 1e-6 * np.abs(kx).sum())


def test_mla_position_zero_identity(orc):
    w = W.mla_workload("zero", 31, [1, 1, 1], [0, 0, 0], num_heads=3, page_size=16,
                       max_seq_len=32, cache_dtype=W.DTYPE_BF16)
    q_out, cache, flags = orc.mla_rope_rmsnorm_quant(w)
    assert flags == 0
    assert np.array_equal(q_out, w.q_rope)
    for t, (row, pos) in _decode_cache_rows(w, cache).items():
        assert pos == 0
        assert np.array_equal(row[512:], w.kv_in[t, 512:])


# ---------------------------------------------------------- through the GQA entry

def _gqa_small(interleaved, mode=None, sec=None, S=32, seed=41, prior=(0, 7, 20), new=(3, 5, 2)):
    return W.gqa_workload("small", seed, list(new), list(prior), num_q_heads=4, num_kv_heads=2,
                          head_size=S, page_size=16, freqs_rows=64, base=10000.0,
                          interleaved=interleaved, position_mode=mode, mrope_section=sec,
                          spare_pages=2)


def _pairs(x, interleaved, S):
    if interleaved:
        return x[..., 0::2], x[..., 1::2]
    return x[..., : S // 2], x[..., S // 2:]


@pytest.mark.parametrize("interleaved", [True, False])
@pytest.mark.parametrize("mode", [None, "ids", "mrope"])
def test_gqa_q_and_k_vs_complex_fp64(orc, interleaved, mode):
    S = 32
    sec = (4, 6, 6) if mode == "mrope" else None
    w = _gqa_small(interleaved, mode, sec, S=S)
    out, cache, flags = orc.qk_rope_paged_ragged(w)
    assert flags == 0
    theta = _theta(S, 10000.0)
    from helpers import expected_slots

    c = w.cache
    slots = expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size)
    v_in = c.view6()
    v_out = cache.reshape(v_in.shape)
    for t, page, row, pos in slots:
        if mode is None:
            pk = np.full(S // 2, pos)
        elif mode == "ids":
            pk = np.full(S // 2, int(w.position_ids[t]))
        else:
            rowsel = np.array([0] * sec[0] + [1] * sec[1] + [2] * sec[2])
            pk = w.position_ids[rowsel, t].astype(np.int64)
        ang = pk * theta
        for src, dst in ((bf16_to_f32(w.q_proj[t]), bf16_to_f32(out[t])),
                         (bf16_to_f32(v_in[page, 0, w.layer_idx, row]),
                          bf16_to_f32(v_out[page, 0, w.layer_idx, row]))):
            a0, a1 = _pairs(src.astype(np.float64), interleaved, S)
            b0, b1 = _pairs(dst.astype(np.float64), interleaved, S)
            e0, e1 = _exact_rotation(a0, a1, np.broadcast_to(ang, a0.shape))
            slack = 1e-6 * (np.abs(a0) + np.abs(a1))
            assert np.all(np.abs(b0 - e0) <= np.abs(e0) * 2.0**-8 + slack)
            assert np.all(np.abs(b1 - e1) <= np.abs(e1) * 2.0**-8 + slack)


def test_gqa_half_split_is_permuted_interleaved(orc):
    S = 32
    w_half = _gqa_small(False, "mrope", (4, 6, 6), S=S)
    w_int = _gqa_small(True, "mrope", (4, 6, 6), S=S)
    # perm maps element k -> 2k and k + S/2 -> 2k + 1
    perm = np.empty(S, np.int64)
    perm[0::2] = np.arange(S // 2)
    perm[1::2] = np.arange(S // 2) + S // 2
    w_int.q_proj = np.ascontiguousarray(w_half.q_proj[..., perm])
    v = w_int.cache.view6()
    v[:, 0] = w_half.cache.view6()[:, 0][..., perm]
    out_h, cache_h, f1 = orc.qk_rope_paged_ragged(w_half)
    out_i, cache_i, f2 = orc.qk_rope_paged_ragged(w_int)
    assert f1 == f2 == 0
    inv = np.argsort(perm)
    assert np.array_equal(out_i[..., inv], out_h)
    ci = cache_i.reshape(v.shape)
    ch = cache_h.reshape(v.shape)
    assert np.array_equal(ci[:, 0][..., inv], ch[:, 0])


def test_gqa_position_ids_equal_slots_is_no_ids(orc):
    from helpers import expected_slots

    w0 = _gqa_small(True, None)
    w1 = _gqa_small(True, "ids")
    c = w0.cache
    pos = np.zeros(w0.T, np.uint32)
    for t, _, _, p in expected_slots(w0.offsets, c.cache_lengths, c.page_table, c.page_size):
        pos[t] = p
    w1.position_ids = pos
    a = orc.qk_rope_paged_ragged(w0)
    b = orc.qk_rope_paged_ragged(w1)
    assert a[2] == b[2] == 0
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gqa_mrope_equal_rows_is_plain_ids(orc):
    w_ids = _gqa_small(False, "ids")
    w_m = _gqa_small(False, "mrope", (4, 6, 6))
    w_m.position_ids = np.stack([w_ids.position_ids] * 3)
    a = orc.qk_rope_paged_ragged(w_ids)
    b = orc.qk_rope_paged_ragged(w_m)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gqa_mrope_single_section_uses_row0(orc):
    w_m = _gqa_small(True, "mrope", (16, 0, 0))
    w_ids = _gqa_small(True, "ids")
    w_ids.position_ids = w_m.position_ids[0].copy()
    w_m.position_ids[1:] = 0xFFFFFFFF  # unused rows are never read
    a = orc.qk_rope_paged_ragged(w_ids)
    b = orc.qk_rope_paged_ragged(w_m)
    assert a[2] == b[2] == 0
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------- GQA with an FP8 K cache

def _gqa_fp8(interleaved=True, mode=None, sec=None, scale=1.0, prior=(0, 7, 20), seed=141):
    return W.gqa_workload("f8", seed, [3, 5, 2], list(prior), num_q_heads=2, num_kv_heads=2,
                          head_size=32, page_size=16, freqs_rows=64, base=10000.0,
                          interleaved=interleaved, position_mode=mode, mrope_section=sec,
                          cache_dtype=W.DTYPE_FP8_E4M3, scale=scale)


def test_gqa_fp8_k_position_zero_is_identity(orc):
    w = _gqa_fp8(prior=(0, 0, 0), seed=142)
    w.offsets = np.array([0, 1, 2, 3], np.uint32)  # one token per request: position 0
    w.q_proj = w.q_proj[:3].copy()
    _, cache, flags = orc.qk_rope_paged_ragged(w, T=3)
    assert flags == 0
    assert np.array_equal(cache, w.cache.data)


@pytest.mark.parametrize("interleaved", [True, False])
def test_gqa_fp8_k_vs_complex_fp64(orc, interleaved):
    from helpers import expected_slots

    S = 32
    w = _gqa_fp8(interleaved)
    out, cache, flags = orc.qk_rope_paged_ragged(w)
    assert flags == 0
    c = w.cache
    theta = _theta(S, 10000.0)
    before, after = c.view6(), c.view6(cache)
    dec = orc.e4m3_decode
    for t, page, row, pos in expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size):
        x = dec(before[page, 0, w.layer_idx, row]).astype(np.float64)
        y = dec(after[page, 0, w.layer_idx, row]).astype(np.float64)
        a0, a1 = _pairs(x, interleaved, S)
        b0, b1 = _pairs(y, interleaved, S)
        e0, e1 = _exact_rotation(a0, a1, np.broadcast_to(pos * theta, a0.shape))
        # one E4M3 rounding: half a step of 2^-3 relative, or 2^-10 absolute (subnormals)
        for b, e in ((b0, e0), (b1, e1)):
            assert np.all(np.abs(b - e) <= np.abs(e) * 2.0**-4 + 2.0**-9 + 1e-6)


def test_gqa_fp8_k_scale_convention(orc):
    """dequantise with the scale, rotate, re-quantise with it: scale 2 on the
    same codes gives the same codes (x2 and /2 are exact)."""
    a = _gqa_fp8(scale=1.0, seed=143)
    b = _gqa_fp8(scale=1.0, seed=143)
    b.cache.scale = 2.0
    _, ca, fa = orc.qk_rope_paged_ragged(a)
    _, cb, fb = orc.qk_rope_paged_ragged(b)
    assert fa == fb == 0 and np.array_equal(ca, cb)
