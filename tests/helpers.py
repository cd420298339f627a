"""Comparison helpers for the tests (independent of both the oracle and the CUDA path)."""
import numpy as np


def bf16_to_f32(h):
    """Exact widening of bf16 bit patterns."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_ordinal(h):
    """Sign-magnitude ordinal of a bf16 pattern (+0 and -0 both map to 0)."""
    h = np.asarray(h, dtype=np.uint16).astype(np.int64)
    mag = h & 0x7FFF
    return np.where(h & 0x8000, -mag, mag)


def e4m3_ordinal(c):
    c = np.asarray(c, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def bf16_ulp_diff(a, b):
    return np.abs(bf16_ordinal(a) - bf16_ordinal(b))


def e4m3_ulp_diff(a, b):
    return np.abs(e4m3_ordinal(a) - e4m3_ordinal(b))


def expected_slots(offsets, cache_lengths, page_table, page_size):
    """Written (token, page, row-in-page, position) by the plain slot formula.

    Token i of request b goes to position cache_lengths[b] + i, which is row
    position % page_size of page page_table[b][position // page_size].
    """
    out = []
    for b in range(len(offsets) - 1):
        for i in range(int(offsets[b + 1]) - int(offsets[b])):
            pos = int(cache_lengths[b]) + i
            page = int(page_table[b][pos // page_size])
            out.append((int(offsets[b]) + i, page, pos % page_size, pos))
    return out
