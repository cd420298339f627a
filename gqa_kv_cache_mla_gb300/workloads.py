"""Seeded synthetic inputs for the fused KV-cache write path.

This module only draws inputs: ragged request lengths, page tables, cache
contents, activations, RMSNorm weights and the precomputed RoPE table that a
serving engine would hand to the three entry points.  It contains none of the
arithmetic of the path itself (no rotation, normalisation or quantisation);
both the CUDA path and the CPU oracle consume exactly the arrays built here.

All arrays are host numpy arrays.  bf16 values are carried as ``uint16`` bit
patterns, FP8 cache bytes as ``uint8``.  The same seed gives the same bytes.

Workloads (sizes and value distributions follow the five benchmark shapes of
the MLA / GQA / K-cache RMSNorm pages):

* ``mla_tiny``     2 requests, new [3,5], prior [0,7], 4 q heads, page 16
* ``mla_decode``   DeepSeek-V3 decode: 256 requests x 1 token, prior U[1,8192]
* ``mla_prefill``  16 requests, new U[512,8192], 1% outliers x20
* ``gqa_llama3``   Llama-3-8B: 32 q / 8 kv heads, head 128, 32 requests
* ``knorm``        8 kv heads, head 128, page 64, 64 mixed decode/prefill requests
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE_UNMAPPED = 0xFFFFFFFF

# cache element types, shared vocabulary with the C ABI enum values
DTYPE_BF16 = 0
DTYPE_FP8_E4M3 = 1
DTYPE_F32 = 2

MLA_KV_NORM_DIM = 512
MLA_ROPE_DIM = 64
MLA_ROW = MLA_KV_NORM_DIM + MLA_ROPE_DIM


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(x) -> np.ndarray:
    """Round fp32 values to bf16 (library cast) and return the uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def e4m3_bits(x) -> np.ndarray:
    """Round fp32 values to FP8 E4M3FN (library cast) and return the codes."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def rope_table(rows: int, dim: int, base: float) -> np.ndarray:
    """Precomputed freqs_cis table, fp32 ``[rows, dim]``.

    Interleaved (cos, sin): entry ``[p, 2i] = cos(p * theta_i)`` and
    ``[p, 2i+1] = sin(p * theta_i)`` with ``theta_i = base ** (-2i / dim)``,
    evaluated in float64 and rounded once to float32.  Plain frequencies, no
    long-context rescaling.
    """
    i = np.arange(dim // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / dim)
    ang = np.arange(rows, dtype=np.float64)[:, None] * theta[None, :]
    tab = np.empty((rows, dim), dtype=np.float64)
    tab[:, 0::2] = np.cos(ang)
    tab[:, 1::2] = np.sin(ang)
    return tab.astype(np.float32)


@dataclasses.dataclass
class PagedCache:
    """Host image of a paged cache plus its addressing metadata.

    Dense layout ``[num_pages, kv_dim, num_layers, page_size, num_heads,
    head_size]`` (kv index 0 is K).  Strides are in elements of ``dtype``.
    """

    data: np.ndarray  # uint16 (bf16) or uint8 (fp8), flat
    dtype: int
    scale: float
    page_table: np.ndarray  # uint32 [B, max_pages_per_seq]
    cache_lengths: np.ndarray  # uint32 [B] prior lengths
    num_pages: int
    kv_dim: int
    num_layers: int
    page_size: int
    num_heads: int
    head_size: int
    custom_strides: Optional[tuple] = None  # (page, kv, layer, token, head), elements

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def strides(self):
        if self.custom_strides is not None:
            return tuple(int(v) for v in self.custom_strides)
        s_head = self.head_size
        s_token = self.num_heads * s_head
        s_layer = self.page_size * s_token
        s_kv = self.num_layers * s_layer
        s_page = self.kv_dim * s_kv
        return (s_page, s_kv, s_layer, s_token, s_head)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == DTYPE_BF16 else 1

    def view6(self, data=None) -> np.ndarray:
        """Logical [pages, kv, layers, page_size, heads, head_size] view of
        ``data`` (default: this cache's bytes) under this cache's strides."""
        d = self.data if data is None else data
        eb = d.itemsize
        shape = (self.num_pages, self.kv_dim, self.num_layers, self.page_size, self.num_heads,
                 self.head_size)
        return np.lib.stride_tricks.as_strided(d, shape=shape,
                                               strides=tuple(eb * v for v in self.strides) + (eb,))


def repad_cache(c: PagedCache, head_pad: int, token_pad: int, rng=None) -> PagedCache:
    """The same logical cache in a padded layout: each head row is followed by
    ``head_pad`` spare elements and each token row by ``token_pad``; spare
    elements hold random bytes."""
    rng = rng_for(12345) if rng is None else rng
    s_head = c.head_size + head_pad
    s_token = c.num_heads * s_head + token_pad
    s_layer = c.page_size * s_token
    s_kv = c.num_layers * s_layer
    s_page = c.kv_dim * s_kv
    n = c.num_pages * s_page
    raw = rng.integers(0, 256, size=n * c.elem_bytes, dtype=np.uint8)
    data = raw.view(np.uint16) if c.elem_bytes == 2 else raw
    out = dataclasses.replace(c, data=data, custom_strides=(s_page, s_kv, s_layer, s_token, s_head))
    out.view6()[...] = c.view6()
    return out


def build_page_table(rng, total_lens, page_size, max_pages_per_seq, whole=False,
                     spare_pages=0):
    """Give request b the pages it needs from one seeded permutation.

    Request b takes ``ceil(total_lens[b] / page_size)`` consecutive entries of
    a random permutation of all pages (``max_pages_per_seq`` entries when
    ``whole``); unused entries hold ``PAGE_UNMAPPED``.  ``spare_pages`` pages
    are allocated but referenced by no request.
    """
    total_lens = np.asarray(total_lens, dtype=np.int64)
    B = total_lens.shape[0]
    if whole:
        need = np.full(B, max_pages_per_seq, dtype=np.int64)
    else:
        need = (total_lens + page_size - 1) // page_size
    assert np.all(need <= max_pages_per_seq)
    num_pages = int(need.sum()) + spare_pages
    perm = rng.permutation(num_pages).astype(np.uint32)
    table = np.full((B, max_pages_per_seq), PAGE_UNMAPPED, dtype=np.uint32)
    cur = 0
    for b in range(B):
        n = int(need[b])
        table[b, :n] = perm[cur:cur + n]
        cur += n
    return table, num_pages


def make_cache(rng, dtype, scale, page_table, cache_lengths, num_pages, kv_dim,
               num_layers, page_size, num_heads, head_size) -> PagedCache:
    """Cache filled with seeded random bytes, so every untouched byte is distinctive."""
    n = num_pages * kv_dim * num_layers * page_size * num_heads * head_size
    eb = 2 if dtype == DTYPE_BF16 else 1
    raw = rng.integers(0, 256, size=n * eb, dtype=np.uint8)
    data = raw.view(np.uint16) if eb == 2 else raw
    return PagedCache(data=data, dtype=dtype, scale=float(scale),
                      page_table=np.ascontiguousarray(page_table, dtype=np.uint32),
                      cache_lengths=np.ascontiguousarray(cache_lengths, dtype=np.uint32),
                      num_pages=num_pages, kv_dim=kv_dim, num_layers=num_layers,
                      page_size=page_size, num_heads=num_heads, head_size=head_size)


def offsets_from_lengths(new_lens) -> np.ndarray:
    off = np.zeros(len(new_lens) + 1, dtype=np.uint32)
    off[1:] = np.cumsum(np.asarray(new_lens, dtype=np.int64))
    return off


def new_slots(offsets, cache_lengths):
    """(token, request, slot position) for every new token: pos = prior + index."""
    out = []
    for b in range(len(offsets) - 1):
        for i in range(int(offsets[b + 1]) - int(offsets[b])):
            out.append((int(offsets[b]) + i, b, int(cache_lengths[b]) + i))
    return out


def normal_bf16(rng, shape, mean=0.0, std=1.0, outlier_frac=0.0, outlier_mult=20.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    if outlier_frac > 0.0:
        mask = rng.random(size=shape, dtype=np.float32) < outlier_frac
        x[mask] *= np.float32(outlier_mult)
    return bf16_bits(x)


def fill_new_k_rows(rng, cache: PagedCache, offsets, layer_idx):
    """Overwrite the K rows of new slots with N(0,1) values (stand-in for a
    QKV GEMM): bf16, or E4M3 codes of N(0,1)/scale for an FP8 cache."""
    v = cache.view6()
    P = cache.page_size
    for t, b, pos in new_slots(offsets, cache.cache_lengths):
        page = int(cache.page_table[b, pos // P])
        shape = (cache.num_heads, cache.head_size)
        if cache.dtype == DTYPE_BF16:
            v[page, 0, layer_idx, pos % P, :, :] = normal_bf16(rng, shape)
        else:
            x = rng.standard_normal(size=shape, dtype=np.float32) / np.float32(cache.scale)
            v[page, 0, layer_idx, pos % P, :, :] = e4m3_bits(x)


@dataclasses.dataclass
class MLAWorkload:
    name: str
    q_rope: np.ndarray  # bf16 bits [T, H, 64]
    kv_in: np.ndarray  # bf16 bits [T, 576]
    offsets: np.ndarray  # uint32 [B+1]
    freqs: np.ndarray  # f32 [rows, 64]
    gamma: np.ndarray  # bf16 bits [512]
    cache: PagedCache
    layer_idx: int
    epsilon: float
    inplace: bool = False  # latent rows already in the cache (in-place variant)
    q_out_dtype: int = DTYPE_BF16

    @property
    def T(self):
        return int(self.q_rope.shape[0])

    @property
    def H(self):
        return int(self.q_rope.shape[1])

    @property
    def B(self):
        return int(self.offsets.shape[0] - 1)


def mla_workload(name, seed, new_lens, prior_lens, num_heads, page_size, max_seq_len,
                 cache_dtype, num_layers=1, layer_idx=0, scale=1.0, outlier_frac=0.0,
                 whole_pages=False, spare_pages=0, epsilon=1e-6) -> MLAWorkload:
    rng = rng_for(seed)
    new_lens = np.asarray(new_lens, dtype=np.int64)
    prior_lens = np.asarray(prior_lens, dtype=np.int64)
    offsets = offsets_from_lengths(new_lens)
    T = int(offsets[-1])
    max_pages = (max_seq_len + page_size - 1) // page_size
    table, num_pages = build_page_table(rng, prior_lens + new_lens, page_size, max_pages,
                                        whole=whole_pages, spare_pages=spare_pages)
    cache = make_cache(rng, cache_dtype, scale, table, prior_lens, num_pages, 1,
                       num_layers, page_size, 1, MLA_ROW)
    q = normal_bf16(rng, (T, num_heads, MLA_ROPE_DIM), outlier_frac=outlier_frac)
    kv = normal_bf16(rng, (T, MLA_ROW), outlier_frac=outlier_frac)
    gamma = normal_bf16(rng, (MLA_KV_NORM_DIM,), mean=1.0, std=0.1)
    freqs = rope_table(max_seq_len, MLA_ROPE_DIM, 10000.0)
    return MLAWorkload(name, q, kv, offsets, freqs, gamma, cache, layer_idx, epsilon)


def place_latent_rows(w: MLAWorkload):
    """Write each new token's 576-wide latent row (w.kv_in) into its cache slot,
    as the latent projection would before the in-place variant runs: bf16
    copied, or E4M3 codes of value / scale (library cast) for an FP8 cache."""
    c = w.cache
    v = c.view6()
    P = c.page_size
    for t, b, pos in new_slots(w.offsets, c.cache_lengths):
        page = int(c.page_table[b, pos // P])
        if c.dtype == DTYPE_BF16:
            v[page, 0, w.layer_idx, pos % P, 0, :] = w.kv_in[t]
        else:
            x = (w.kv_in[t].astype(np.uint32) << 16).view(np.float32) / np.float32(c.scale)
            v[page, 0, w.layer_idx, pos % P, 0, :] = e4m3_bits(x)


def context_offsets(cache: PagedCache, offsets) -> np.ndarray:
    """Ragged offsets over whole contexts (prior + new tokens per request)."""
    new = np.diff(np.asarray(offsets, dtype=np.int64))
    return offsets_from_lengths(np.asarray(cache.cache_lengths, dtype=np.int64) + new)


def mla_inplace(w: MLAWorkload) -> MLAWorkload:
    """The same step for the in-place variant: latent rows placed in the cache."""
    place_latent_rows(w)
    w.inplace = True
    return w


def fill_contexts(rng, cache: PagedCache, offsets, layer_idx):
    """N(0,1) latent rows (bf16, or E4M3 codes of value / scale) in every
    context slot (prior and new tokens) of every request."""
    ctx = context_offsets(cache, offsets)
    v = cache.view6()
    P = cache.page_size
    for b in range(len(ctx) - 1):
        n = int(ctx[b + 1]) - int(ctx[b])
        if n == 0:
            continue
        x = rng.standard_normal(size=(n, cache.head_size), dtype=np.float32)
        rows = bf16_bits(x) if cache.dtype == DTYPE_BF16 else e4m3_bits(x / np.float32(cache.scale))
        for p in range(n):
            v[int(cache.page_table[b, p // P]), 0, layer_idx, p % P, 0, :] = rows[p]
    return ctx


@dataclasses.dataclass
class GatherWorkload:
    name: str
    cache: PagedCache
    layer_idx: int
    ctx_offsets: np.ndarray  # uint32 [B+1] over whole contexts
    out_dtype: int
    out_scale: float
    dynamic: bool = False  # per-row dynamic FP8 (codes + one scale per row)

    @property
    def rows(self):
        return int(self.ctx_offsets[-1])

    @property
    def T(self):
        return self.rows


def mla_gather(w: MLAWorkload, out_dtype=DTYPE_FP8_E4M3, out_scale=1.0, seed=9,
               dynamic=False) -> GatherWorkload:
    ctx = fill_contexts(rng_for(seed), w.cache, w.offsets, w.layer_idx)
    return GatherWorkload(w.name + "_gather", w.cache, w.layer_idx, ctx,
                          DTYPE_FP8_E4M3 if dynamic else out_dtype, out_scale, dynamic)


@dataclasses.dataclass
class ConvertWorkload:
    name: str
    x: np.ndarray  # bf16 bits, flat (convert) or [rows, cols] (per-row quantisation)
    scale: float = 1.0
    per_row: bool = False

    @property
    def T(self):
        return int(self.x.shape[0]) if self.per_row else int(self.x.size)


def fp8_convert(n=1 << 26, seed=10, scale=1.0) -> ConvertWorkload:
    """bf16 weights N(0, 0.05) (n values) to E4M3."""
    return ConvertWorkload("fp8_convert", normal_bf16(rng_for(seed), (n,), std=0.05), scale)


def fp8_quant_rows(rows=32768, cols=2048, seed=11) -> ConvertWorkload:
    """Per-token dynamic FP8 of activations: rows of N(0,1) with 1% outliers x20."""
    x = normal_bf16(rng_for(seed), (rows, cols), outlier_frac=0.01)
    return ConvertWorkload("fp8_quant_rows", x, 1.0, per_row=True)


def mla_tiny(cache_dtype=DTYPE_BF16, seed=1) -> MLAWorkload:
    """2 requests, new [3,5], prior [0,7], 4 q heads, page 16, max_seq 64, 8 pages."""
    return mla_workload("mla_tiny", seed, [3, 5], [0, 7], num_heads=4, page_size=16,
                        max_seq_len=64, cache_dtype=cache_dtype, num_layers=2,
                        layer_idx=1, whole_pages=True)


def mla_decode(cache_dtype=DTYPE_FP8_E4M3, seed=2, num_requests=256) -> MLAWorkload:
    """DeepSeek-V3 decode: 256 x 1 new token, prior U[1,8192], 128 q heads, page 128."""
    rng = rng_for(seed + 1000)
    prior = rng.integers(1, 8192, size=num_requests, endpoint=True)
    return mla_workload("mla_decode", seed, np.ones(num_requests, np.int64), prior,
                        num_heads=128, page_size=128, max_seq_len=16384,
                        cache_dtype=cache_dtype)


def mla_prefill(cache_dtype=DTYPE_BF16, seed=3, num_requests=16) -> MLAWorkload:
    """Ragged prefill: 16 requests, new U[512,8192], prior 0, 1% outliers x20."""
    rng = rng_for(seed + 1000)
    new = rng.integers(512, 8192, size=num_requests, endpoint=True)
    return mla_workload("mla_prefill", seed, new, np.zeros(num_requests, np.int64),
                        num_heads=128, page_size=128, max_seq_len=16384,
                        cache_dtype=cache_dtype, outlier_frac=0.01)


@dataclasses.dataclass
class GQAWorkload:
    name: str
    q_proj: np.ndarray  # bf16 bits [T, Hq, S]
    offsets: np.ndarray
    freqs: np.ndarray  # f32 [rows, S]
    position_ids: Optional[np.ndarray]  # uint32 [T] or [3, T]
    mrope_section: Optional[np.ndarray]  # uint32 [3]
    interleaved: bool
    cache: PagedCache
    layer_idx: int

    @property
    def T(self):
        return int(self.q_proj.shape[0])

    @property
    def B(self):
        return int(self.offsets.shape[0] - 1)


def gqa_workload(name, seed, new_lens, prior_lens, num_q_heads, num_kv_heads, head_size,
                 page_size, freqs_rows, base, interleaved, position_mode=None,
                 mrope_section=None, num_layers=2, layer_idx=1, spare_pages=0,
                 pos_limit=None, cache_dtype=DTYPE_BF16, scale=1.0) -> GQAWorkload:
    """position_mode: None (slot positions), "ids" ([T]) or "mrope" ([3, T])."""
    rng = rng_for(seed)
    new_lens = np.asarray(new_lens, dtype=np.int64)
    prior_lens = np.asarray(prior_lens, dtype=np.int64)
    offsets = offsets_from_lengths(new_lens)
    T = int(offsets[-1])
    total = prior_lens + new_lens
    max_pages = int(max(1, (int(total.max()) + page_size - 1) // page_size)) if len(total) else 1
    table, num_pages = build_page_table(rng, total, page_size, max_pages,
                                        spare_pages=spare_pages)
    cache = make_cache(rng, cache_dtype, scale, table, prior_lens, num_pages, 2, num_layers,
                       page_size, num_kv_heads, head_size)
    fill_new_k_rows(rng, cache, offsets, layer_idx)
    q = normal_bf16(rng, (T, num_q_heads, head_size))
    lim = freqs_rows if pos_limit is None else pos_limit
    pos_ids = None
    sec = None
    if position_mode == "ids":
        pos_ids = rng.integers(0, lim, size=T, dtype=np.uint32)
    elif position_mode == "mrope":
        pos_ids = rng.integers(0, lim, size=(3, T), dtype=np.uint32)
        sec = np.asarray(mrope_section, dtype=np.uint32)
    freqs = rope_table(freqs_rows, head_size, base)
    return GQAWorkload(name, q, offsets, freqs, pos_ids, sec, bool(interleaved), cache,
                       layer_idx)


def gqa_llama3(interleaved=True, position_mode=None, seed=4, num_requests=32,
               cache_dtype=DTYPE_BF16, scale=1.0) -> GQAWorkload:
    """Llama-3-8B: 32 q / 8 kv heads, head 128, new U[1,2048], prior U[0,4096], page 128."""
    rng = rng_for(seed + 1000)
    new = rng.integers(1, 2048, size=num_requests, endpoint=True)
    prior = rng.integers(0, 4096, size=num_requests, endpoint=True)
    sec = (16, 24, 24) if position_mode == "mrope" else None
    return gqa_workload("gqa_llama3", seed, new, prior, 32, 8, 128, 128, 8192, 500000.0,
                        interleaved, position_mode=position_mode, mrope_section=sec,
                        cache_dtype=cache_dtype, scale=scale)


@dataclasses.dataclass
class KNormWorkload:
    name: str
    offsets: np.ndarray
    gamma: np.ndarray  # bf16 bits [G]
    epsilon: float
    weight_offset: float
    multiply_before_cast: bool
    cache: PagedCache
    layer_idx: int
    per_head_norm: bool = True

    @property
    def T(self):
        return int(self.offsets[-1])

    @property
    def B(self):
        return int(self.offsets.shape[0] - 1)


def knorm_workload(name, seed, new_lens, prior_lens, num_kv_heads, head_size, page_size,
                   gamma_len, weight_offset=0.0, multiply_before_cast=True, num_layers=2,
                   layer_idx=1, spare_pages=0, epsilon=1e-6, per_head_norm=True) -> KNormWorkload:
    rng = rng_for(seed)
    new_lens = np.asarray(new_lens, dtype=np.int64)
    prior_lens = np.asarray(prior_lens, dtype=np.int64)
    offsets = offsets_from_lengths(new_lens)
    total = prior_lens + new_lens
    max_pages = int(max(1, (int(total.max()) + page_size - 1) // page_size)) if len(total) else 1
    table, num_pages = build_page_table(rng, total, page_size, max_pages,
                                        spare_pages=spare_pages)
    cache = make_cache(rng, DTYPE_BF16, 1.0, table, prior_lens, num_pages, 2, num_layers,
                       page_size, num_kv_heads, head_size)
    fill_new_k_rows(rng, cache, offsets, layer_idx)
    gamma = normal_bf16(rng, (gamma_len,), mean=1.0, std=0.1)
    return KNormWorkload(name, offsets, gamma, epsilon, float(weight_offset),
                         bool(multiply_before_cast), cache, layer_idx, bool(per_head_norm))


def knorm_paged(gamma_len=128, seed=5, num_requests=64, weight_offset=0.0,
                multiply_before_cast=True, per_head_norm=True) -> KNormWorkload:
    """8 kv heads, head 128, page 64; each request decode (p=0.5) or prefill U[64,1024]."""
    rng = rng_for(seed + 1000)
    decode = rng.random(num_requests) < 0.5
    pre = rng.integers(64, 1024, size=num_requests, endpoint=True)
    new = np.where(decode, 1, pre)
    prior = rng.integers(0, 2048, size=num_requests, endpoint=True)
    return knorm_workload("knorm", seed, new, prior, 8, 128, 64, gamma_len,
                          weight_offset=weight_offset, multiply_before_cast=multiply_before_cast,
                          per_head_norm=per_head_norm)


def algorithmic_bytes_mla(T, H, cache_dtype, distinct_positions=None):
    """Bytes each launch must move: q in+out, kv row in, cache row out, freqs rows."""
    c = 2 if cache_dtype == DTYPE_BF16 else 1
    rows = T if distinct_positions is None else distinct_positions
    return T * (2 * H * MLA_ROPE_DIM * 2 + MLA_ROW * 2 + MLA_ROW * c) + rows * MLA_ROPE_DIM * 4


def algorithmic_bytes_gqa(T, Hq, Hk, S, distinct_rows, k_bytes=2):
    return T * (2 * Hq * S * 2 + 2 * Hk * S * k_bytes) + distinct_rows * S * 4


def algorithmic_bytes_knorm(T, Hk, G):
    return T * 2 * Hk * G * 2


# Benchmark workloads: name -> (builder(seed), kernel source file, description).
REGISTRY = {
    # name: (builder, kernel source, description)
    "mla_decode": (lambda s: mla_decode(DTYPE_FP8_E4M3, seed=s), "mla_rope_rmsnorm_quant.cu",
                   "MLA decode DeepSeek-V3: 256 req x 1 token, prior U[1,8192], H=128, "
                   "512+64, page 128, FP8 E4M3 cache (scale 1.0)"),
    "mla_decode_bf16": (lambda s: mla_decode(DTYPE_BF16, seed=s), "mla_rope_rmsnorm_quant.cu",
                        "MLA decode DeepSeek-V3, bf16 cache"),
    "mla_prefill_bf16": (lambda s: mla_prefill(DTYPE_BF16, seed=s + 1),
                         "mla_rope_rmsnorm_quant.cu",
                         "MLA ragged prefill: 16 req, new U[512,8192], H=128, 1% outliers x20, "
                         "bf16 cache"),
    "mla_prefill_fp8": (lambda s: mla_prefill(DTYPE_FP8_E4M3, seed=s + 1),
                        "mla_rope_rmsnorm_quant.cu",
                        "MLA ragged prefill: 16 req, new U[512,8192], H=128, 1% outliers x20, "
                        "FP8 E4M3 cache"),
    "mla_decode_fp8q": (lambda s: dataclasses.replace(mla_decode(DTYPE_FP8_E4M3, seed=s),
                                                      q_out_dtype=DTYPE_FP8_E4M3),
                        "mla_rope_rmsnorm_quant.cu",
                        "MLA decode DeepSeek-V3, FP8 cache and FP8 q_rope output"),
    "mla_decode_inplace": (lambda s: mla_inplace(mla_decode(DTYPE_FP8_E4M3, seed=s)),
                           "mla_rope_rmsnorm_quant.cu",
                           "MLA decode DeepSeek-V3, in-place variant on an FP8 cache"),
    "mla_prefill_inplace": (lambda s: mla_inplace(mla_prefill(DTYPE_BF16, seed=s + 1)),
                            "mla_rope_rmsnorm_quant.cu",
                            "MLA ragged prefill, in-place variant on a bf16 cache"),
    "mla_gather_prefill": (lambda s: mla_gather(mla_prefill(DTYPE_BF16, seed=s + 1)),
                           "mla_gather_latent.cu",
                           "paged->contiguous latent gather of the prefill contexts, bf16 "
                           "cache to FP8 E4M3 (scale 1)"),
    "mla_gather_prefill_dynamic": (lambda s: mla_gather(mla_prefill(DTYPE_BF16, seed=s + 1),
                                                       dynamic=True),
                                   "mla_gather_latent.cu",
                                   "paged->contiguous latent gather of the prefill contexts, bf16 "
                                   "cache to FP8 E4M3 with a dynamic scale per row"),
    "fp8_convert": (lambda s: fp8_convert(seed=s + 10), "fp8_codec.cu",
                    "bf16 -> E4M3 conversion of 2^26 values"),
    "fp8_quant_rows": (lambda s: fp8_quant_rows(seed=s + 11), "fp8_codec.cu",
                       "per-row dynamic FP8 of a [32768, 2048] bf16 activation"),
    "mla_prefill_bf16_4req": (lambda s: mla_prefill(DTYPE_BF16, seed=s + 1, num_requests=4),
                              "mla_rope_rmsnorm_quant.cu",
                              "MLA ragged prefill, 4 of the 16 requests (profiling size), bf16 cache"),
    "mla_prefill_fp8_4req": (lambda s: mla_prefill(DTYPE_FP8_E4M3, seed=s + 1, num_requests=4),
                             "mla_rope_rmsnorm_quant.cu",
                             "MLA ragged prefill, 4 of the 16 requests (profiling size), FP8 cache"),
    "mla_prefill_inplace_4req": (lambda s: mla_inplace(mla_prefill(DTYPE_BF16, seed=s + 1,
                                                                    num_requests=4)),
                                 "mla_rope_rmsnorm_quant.cu",
                                 "MLA ragged prefill in place, 4 of the 16 requests (profiling "
                                 "size), bf16 cache"),
    "gqa_interleaved": (lambda s: gqa_llama3(True, None, seed=s + 2), "qk_rope_paged_ragged.cu",
                        "GQA Llama-3-8B Q/K RoPE, interleaved, slot positions"),
    "gqa_half_ids": (lambda s: gqa_llama3(False, "ids", seed=s + 2), "qk_rope_paged_ragged.cu",
                     "GQA Llama-3-8B Q/K RoPE, half-split, position_ids"),
    "gqa_mrope": (lambda s: gqa_llama3(False, "mrope", seed=s + 2), "qk_rope_paged_ragged.cu",
                  "GQA Llama-3-8B Q/K RoPE, half-split, mrope (16,24,24)"),
    "gqa_fp8k": (lambda s: gqa_llama3(True, None, seed=s + 2, cache_dtype=DTYPE_FP8_E4M3),
                 "qk_rope_paged_ragged.cu",
                 "GQA Llama-3-8B Q/K RoPE, interleaved, FP8 E4M3 K cache (scale 1.0)"),
    "knorm128": (lambda s: knorm_paged(128, seed=s + 3), "rms_norm_kv_cache_paged.cu",
                 "paged K-cache RMSNorm: 8 kv heads x 128, page 64, 64 mixed requests, G=128"),
    "knorm128_cast_first": (lambda s: knorm_paged(128, seed=s + 3, weight_offset=0.5,
                                                  multiply_before_cast=False),
                            "rms_norm_kv_cache_paged.cu",
                            "paged K-cache RMSNorm, G=128, multiply_before_cast=false, "
                            "weight_offset=0.5"),
    "knorm_whole_row": (lambda s: knorm_paged(1024, seed=s + 3, per_head_norm=False),
                        "rms_norm_kv_cache_paged.cu",
                        "paged K-cache RMSNorm over the whole 8x128 K row (per_head_norm=false)"),
    "knorm64": (lambda s: knorm_paged(64, seed=s + 3), "rms_norm_kv_cache_paged.cu",
                "paged K-cache RMSNorm: 8 kv heads x 128, page 64, 64 mixed requests, "
                "subset G=64"),
}


def ceil_div(a, b):
    return (a + b - 1) // b


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("annotations", "math")]
