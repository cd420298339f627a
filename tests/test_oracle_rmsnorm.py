"""Pins for the oracle's RMSNorm steps (MLA latent part and in-place K norm).

Closed forms: with unit weights the output's root-mean-square equals
sqrt(ms / (ms + eps)), ms = mean(x^2); with eps = 0 the output is invariant
to scaling x by a power of two.  Library special case:
torch.nn.functional.rms_norm.
"""
import numpy as np
import pytest
import torch

from gqa_kv_cache_mla_gb300 import workloads as W
from helpers import bf16_to_f32, bf16_ulp_diff, expected_slots


def _torch_rms_norm64(x, w, eps):
    x = torch.from_numpy(np.array(x, dtype=np.float64))
    w = torch.from_numpy(np.array(w, dtype=np.float64))
    return torch.nn.functional.rms_norm(x, (x.shape[-1],), weight=w, eps=eps).numpy()


@pytest.mark.parametrize("n", [512, 128, 64, 96, 7])
@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_unit_weight_rms_closed_form(orc, n, eps):
    rng = np.random.default_rng(51 + n)
    for _ in range(50):
        x = (rng.standard_normal(n) * rng.uniform(0.1, 10)).astype(np.float32)
        y = orc.rms_norm_f32(x, np.ones(n, np.float32), eps).astype(np.float64)
        ms = np.mean(x.astype(np.float64) ** 2)
        want = np.sqrt(ms / (ms + eps))
        got = np.sqrt(np.mean(y**2))
        assert abs(got - want) <= 1e-5 * want


def test_power_of_two_scale_invariance(orc):
    rng = np.random.default_rng(52)
    for n in (512, 128, 64):
        x = rng.standard_normal(n).astype(np.float32)
        w = (1 + 0.1 * rng.standard_normal(n)).astype(np.float32)
        y = orc.rms_norm_f32(x, w, 0.0)
        for k in (-3, 1, 5):
            y2 = orc.rms_norm_f32(x * np.float32(2.0**k), w, 0.0)
            assert np.array_equal(y, y2)


def test_rms_norm_vs_torch(orc):
    rng = np.random.default_rng(53)
    for n in (512, 128, 64):
        for _ in range(100):
            x = (rng.standard_normal(n) * 3).astype(np.float32)
            w = (1 + 0.1 * rng.standard_normal(n)).astype(np.float32)
            y = orc.rms_norm_f32(x, w, 1e-6).astype(np.float64)
            ref = _torch_rms_norm64(x, w, 1e-6)
            assert np.all(np.abs(y - ref) <= 16 * 2.0**-24 * np.abs(ref) + 1e-12)


def test_mla_latent_part_vs_torch(orc):
    w = W.mla_tiny()
    _, cache, flags = orc.mla_rope_rmsnorm_quant(w)
    assert flags == 0
    c = w.cache
    v = cache.reshape(c.view6().shape)
    g = bf16_to_f32(w.gamma)
    for t, page, row, pos in expected_slots(w.offsets, c.cache_lengths, c.page_table,
                                            c.page_size):
        got = v[page, 0, w.layer_idx, row, 0, :512]
        ref = _torch_rms_norm64(bf16_to_f32(w.kv_in[t, :512]), g, w.epsilon)
        ref_bits = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)
        assert bf16_ulp_diff(got, ref_bits).max() <= 1


def _knorm_small(G, per_head=True, wo=0.0, mbc=True, seed=61, S=32, Hk=3):
    return W.knorm_workload("small", seed, [3, 1, 6], [0, 9, 17], num_kv_heads=Hk,
                            head_size=S, page_size=8, gamma_len=G, weight_offset=wo,
                            multiply_before_cast=mbc, spare_pages=2)


@pytest.mark.parametrize("G", [32, 16, 8, 5])
def test_knorm_subset_vs_torch(orc, G):
    w = _knorm_small(G)
    cache, flags = orc.rms_norm_kv_cache_paged(w)
    assert flags == 0
    c = w.cache
    before = c.view6()
    after = cache.reshape(before.shape)
    g = bf16_to_f32(w.gamma)
    for t, page, row, pos in expected_slots(w.offsets, c.cache_lengths, c.page_table,
                                            c.page_size):
        for h in range(c.num_heads):
            x = bf16_to_f32(before[page, 0, w.layer_idx, row, h, :G])
            ref = _torch_rms_norm64(x, g, w.epsilon).astype(np.float32)
            ref_bits = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(
                np.uint16)
            assert bf16_ulp_diff(after[page, 0, w.layer_idx, row, h, :G], ref_bits).max() <= 1
            # columns past the gamma length are not touched
            assert np.array_equal(after[page, 0, w.layer_idx, row, h, G:],
                                  before[page, 0, w.layer_idx, row, h, G:])


def test_knorm_weight_offset_adds_to_gamma(orc):
    w1 = _knorm_small(32)
    w2 = _knorm_small(32, wo=1.0)
    w1.gamma = W.bf16_bits(np.ones(32, np.float32))
    w2.gamma = W.bf16_bits(np.zeros(32, np.float32))
    a, fa = orc.rms_norm_kv_cache_paged(w1)
    b, fb = orc.rms_norm_kv_cache_paged(w2)
    assert fa == fb == 0
    assert np.array_equal(a, b)
    w3 = _knorm_small(32, wo=0.25)
    w3.gamma = W.bf16_bits(np.full(32, 0.75, np.float32))
    c3, _ = orc.rms_norm_kv_cache_paged(w3)
    assert np.array_equal(a, c3)


def test_knorm_multiply_after_cast_within_one_ulp(orc):
    """multiply_before_cast=False (parity unpinned): two roundings instead of one."""
    a, _ = orc.rms_norm_kv_cache_paged(_knorm_small(32, mbc=True))
    b, _ = orc.rms_norm_kv_cache_paged(_knorm_small(32, mbc=False))
    assert bf16_ulp_diff(a, b).max() <= 1
    assert not np.array_equal(a, b)


def test_knorm_whole_row_norm(orc):
    """per_head_norm=False (parity unpinned): one norm over all heads of a token."""
    Hk, S = 3, 32
    w = _knorm_small(Hk * S, per_head=False)
    cache, flags = orc.rms_norm_kv_cache_paged(w, per_head_norm=False)
    assert flags == 0
    c = w.cache
    before = c.view6()
    after = cache.reshape(before.shape)
    g = bf16_to_f32(w.gamma)
    for t, page, row, pos in expected_slots(w.offsets, c.cache_lengths, c.page_table,
                                            c.page_size):
        x = bf16_to_f32(before[page, 0, w.layer_idx, row].reshape(-1))
        ref = _torch_rms_norm64(x, g, w.epsilon).astype(np.float32)
        ref_bits = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(
            np.uint16)
        assert bf16_ulp_diff(after[page, 0, w.layer_idx, row].reshape(-1), ref_bits).max() <= 1


@pytest.mark.parametrize("gamma_value,wo", [(1.0, 0.0), (2.0, 0.0), (0.25, 0.75), (0.5, -0.25)])
def test_knorm_cast_first_reduces_to_one_rounding_for_power_of_two_weights(orc, gamma_value, wo):
    """multiply_before_cast=False rounds x*r to bf16 and then multiplies by
    w = gamma + weight_offset; when w is a power of two that product is exact,
    so the two orders give the same bits."""
    a = _knorm_small(32, mbc=True, wo=wo)
    b = _knorm_small(32, mbc=False, wo=wo)
    for w in (a, b):
        w.gamma = np.full_like(w.gamma, W.bf16_bits(np.float32(gamma_value)))
    ca, _ = orc.rms_norm_kv_cache_paged(a)
    cb, _ = orc.rms_norm_kv_cache_paged(b)
    assert np.array_equal(ca, cb)
