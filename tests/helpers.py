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


def expected_slots(offsets, cache_lengths, page_table, page_size, num_pages=None):
    """Written (token, page, row-in-page, position) by the plain slot formula.

    Token i of request b goes to position cache_lengths[b] + i, which is row
    position % page_size of page page_table[b][position // page_size].  With
    ``num_pages``, slots that map to no valid page are left out.
    """
    out = []
    for b in range(len(offsets) - 1):
        for i in range(int(offsets[b + 1]) - int(offsets[b])):
            pos = int(cache_lengths[b]) + i
            if pos // page_size >= page_table.shape[-1]:
                continue
            page = int(page_table[b][pos // page_size])
            if num_pages is not None and page >= num_pages:
                continue
            out.append((int(offsets[b]) + i, page, pos % page_size, pos))
    return out


def written_row_mask(cache, slots, layer_idx):
    """Boolean [num_pages, num_layers, page_size] of K rows the call may write."""
    m = np.zeros((cache.num_pages, cache.num_layers, cache.page_size), dtype=bool)
    for _, page, row, _ in slots:
        m[page, layer_idx, row] = True
    return m


def compare_cache(cache, gpu, ref, slots, layer_idx, fp8, max_ulp_frac=None, cols=None,
                  bf16_max_ulp=1):
    """GPU cache vs oracle cache.

    Elements outside the rows the call writes (and, with ``cols``, columns at
    or past ``cols``) must be bit-identical; inside, bf16 may differ by 1 ulp
    and FP8 by 1 ulp on at most ``max_ulp_frac`` of the written elements.
    ``bf16_max_ulp`` > 1 (for results rounded twice) allows differences up to
    that many ulp on at most 1e-3 of the written elements.
    Returns the number of differing elements.
    """
    gpu = gpu.reshape(-1)
    ref = ref.reshape(-1)
    diff = np.flatnonzero(gpu != ref)
    if diff.size == 0:
        return 0
    if cache.custom_strides is None:
        shape = (cache.num_pages, cache.kv_dim, cache.num_layers, cache.page_size,
                 cache.num_heads, cache.head_size)
        page, kv, layer, row, head, col = np.unravel_index(diff, shape)
        mask = written_row_mask(cache, slots, layer_idx)
        inside = (kv == 0) & mask[page, layer, row]
        if cols is not None:
            inside &= col < cols
    else:  # padded layout (small caches only): flat indices of the writable elements
        flat = cache.view6(np.arange(gpu.size, dtype=np.int64))
        allowed = np.zeros(gpu.size, dtype=bool)
        for _, page, row, _ in slots:
            allowed[flat[page, 0, layer_idx, row, :, : (cols or cache.head_size)].reshape(-1)] = True
        inside = allowed[diff]
    assert inside.all(), "bytes changed outside the written rows: %d" % int((~inside).sum())
    if fp8:
        u = e4m3_ulp_diff(gpu[diff], ref[diff])
        assert u.max() <= 1, "fp8 difference above 1 ulp: %d" % int(u.max())
        n_written = len(slots) * cache.num_heads * (cols or cache.head_size)
        frac = diff.size / max(1, n_written)
        assert frac <= (max_ulp_frac if max_ulp_frac is not None else 1e-3), frac
    else:
        u = bf16_ulp_diff(gpu[diff], ref[diff])
        assert u.max() <= bf16_max_ulp, "bf16 difference above %d ulp: %d" % (bf16_max_ulp,
                                                                             int(u.max()))
        n_written = len(slots) * cache.num_heads * (cols or cache.head_size)
        assert (u > 1).sum() <= max(1.0, 1e-3 * n_written), int((u > 1).sum())
    return int(diff.size)


def compare_bf16(gpu, ref, max_ulp=1):
    """bf16 bit patterns equal within ``max_ulp`` ulp (+0 and -0 count as equal).

    Raises AssertionError on a larger difference; returns the number of
    elements whose ordinals differ (0 when every value matches).
    """
    gpu = np.asarray(gpu, dtype=np.uint16).reshape(-1)
    ref = np.asarray(ref, dtype=np.uint16).reshape(-1)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    diff = np.flatnonzero(gpu != ref)
    if diff.size == 0:
        return 0
    u = bf16_ulp_diff(gpu[diff], ref[diff])
    assert u.max() <= max_ulp, "bf16 difference above %d ulp: %d" % (max_ulp, int(u.max()))
    return int((u > 0).sum())


def compare_e4m3(gpu, ref, max_frac=1e-3):
    """E4M3 codes equal except 1-ulp flips on at most max_frac of them."""
    gpu = np.asarray(gpu).reshape(-1)
    ref = np.asarray(ref).reshape(-1)
    diff = np.flatnonzero(gpu != ref)
    if diff.size:
        u = e4m3_ulp_diff(gpu[diff], ref[diff])
        assert u.max() <= 1, "fp8 difference above 1 ulp: %d" % int(u.max())
        assert diff.size <= max(1, max_frac * gpu.size), diff.size / gpu.size
    return int(diff.size)
