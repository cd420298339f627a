"""The comparison helpers the parity tests use, checked on hand-made patterns (CPU).

The parity bar: bf16 results within 1 bf16 ulp of the oracle's fp32 result
rounded to bf16 (sign-magnitude ordinal distance, +0 equal to -0); FP8 E4M3
results within 1 ulp on at most 0.1% of the elements; bytes outside the
written rows bit-identical.
"""
import numpy as np
import pytest

from gqa_kv_cache_mla_gb300 import workloads as W
from helpers import (bf16_ulp_diff, compare_bf16, compare_cache, compare_e4m3,
                     e4m3_ulp_diff, expected_slots)

# bf16 patterns: 1.0 and its next two successors; -0 and +0
ONE, ONE_P1, ONE_P2 = 0x3F80, 0x3F81, 0x3F82
NEG_ZERO, POS_ZERO = 0x8000, 0x0000


def test_bf16_equal_passes():
    a = np.array([ONE, POS_ZERO, 0x7F7F, 0xC2F7], np.uint16)
    assert compare_bf16(a, a.copy()) == 0


def test_bf16_one_ulp_passes_and_counts():
    a = np.array([ONE, ONE, 0xC000, 0x1234], np.uint16)
    b = np.array([ONE_P1, ONE, 0xC001, 0x1234], np.uint16)
    assert compare_bf16(a, b) == 2


def test_bf16_two_ulp_fails():
    a = np.array([ONE, ONE], np.uint16)
    b = np.array([ONE_P2, ONE], np.uint16)
    with pytest.raises(AssertionError):
        compare_bf16(a, b)
    assert compare_bf16(a, b, max_ulp=2) == 1


def test_bf16_signed_zeros_equal():
    a = np.array([NEG_ZERO, POS_ZERO], np.uint16)
    b = np.array([POS_ZERO, NEG_ZERO], np.uint16)
    assert compare_bf16(a, b) == 0
    assert bf16_ulp_diff(np.uint16(NEG_ZERO), np.uint16(POS_ZERO)) == 0


def test_bf16_across_zero_is_distance_of_magnitudes():
    # smallest positive subnormal vs smallest negative subnormal: 2 ulp apart
    assert bf16_ulp_diff(np.uint16(0x0001), np.uint16(0x8001)) == 2
    with pytest.raises(AssertionError):
        compare_bf16(np.array([0x0001], np.uint16), np.array([0x8001], np.uint16))


def test_bf16_shape_mismatch_fails():
    with pytest.raises(AssertionError):
        compare_bf16(np.zeros(3, np.uint16), np.zeros(4, np.uint16))


def test_e4m3_fraction_and_distance():
    ref = np.full(10000, 0x38, np.uint8)  # 1.0
    gpu = ref.copy()
    gpu[:10] = 0x39  # 10 one-ulp flips = 0.1%
    assert compare_e4m3(gpu, ref) == 10
    gpu[10] = 0x39  # 11 > 0.1%
    with pytest.raises(AssertionError):
        compare_e4m3(gpu, ref)
    two = ref.copy()
    two[0] = 0x3A
    with pytest.raises(AssertionError):
        compare_e4m3(two, ref)
    assert e4m3_ulp_diff(np.uint8(0x80), np.uint8(0x00)) == 0


def _tiny_cache(dtype):
    w = W.mla_tiny(cache_dtype=dtype)
    c = w.cache
    slots = expected_slots(w.offsets, c.cache_lengths, c.page_table, c.page_size)
    return w, c, slots


def test_cache_compare_outside_rows_fails():
    w, c, slots = _tiny_cache(W.DTYPE_BF16)
    ref = c.data.copy()
    gpu = ref.copy()
    # flat element 0 is in layer 0; the tiny workload writes layer 1 only
    assert w.layer_idx != 0
    gpu.reshape(-1)[0] ^= 1
    with pytest.raises(AssertionError):
        compare_cache(c, gpu, ref, slots, w.layer_idx, fp8=False)


def test_cache_compare_inside_rows_tolerance():
    w, c, slots = _tiny_cache(W.DTYPE_BF16)
    ref = c.data.copy()
    v6 = c.view6(ref)
    _, page, row, _ = slots[0]
    v6[page, 0, w.layer_idx, row, 0, 0] = ONE
    gpu = ref.copy()
    c.view6(gpu)[page, 0, w.layer_idx, row, 0, 0] = ONE_P1
    assert compare_cache(c, gpu, ref, slots, w.layer_idx, fp8=False) == 1
    c.view6(gpu)[page, 0, w.layer_idx, row, 0, 0] = ONE_P2
    with pytest.raises(AssertionError):
        compare_cache(c, gpu, ref, slots, w.layer_idx, fp8=False)


def test_cache_compare_fp8_fraction():
    w, c, slots = _tiny_cache(W.DTYPE_FP8_E4M3)
    ref = c.data.copy()
    _, page, row, _ = slots[0]
    c.view6(ref)[page, 0, w.layer_idx, row, 0, :] = 0x38
    gpu = ref.copy()
    # 8 rows x 576 written values: 4 flips is 0.087% (passes), 5 is 0.11% (fails)
    c.view6(gpu)[page, 0, w.layer_idx, row, 0, :4] = 0x39
    assert compare_cache(c, gpu, ref, slots, w.layer_idx, fp8=True) == 4
    c.view6(gpu)[page, 0, w.layer_idx, row, 0, 4] = 0x39
    with pytest.raises(AssertionError):
        compare_cache(c, gpu, ref, slots, w.layer_idx, fp8=True)
