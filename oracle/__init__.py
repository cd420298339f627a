"""ctypes front end of the CPU oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the benchmark's CPU-baseline leg, never by the product path.  The C
file is compiled with gcc (fp32, ``-ffp-contract=off``, OpenMP when the
compiler has it) into ``oracle/liboracle.so``; nothing here touches CUDA.

Every function takes and returns host numpy arrays: bf16 as uint16 bit
patterns, FP8 E4M3 as uint8, positions and offsets as uint32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None
_libpath = _LIB

FLAG_PAGE = 1
FLAG_POS = 2
FLAG_OFFSETS = 4


def compile_source(src: str, out: str) -> str:
    """gcc the oracle source ``src`` into the shared library ``out``."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wno-unknown-pragmas", "-Wno-maybe-uninitialized"]
    tmp = out + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", src, "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle (a second or two).  Returns the library path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return compile_source(_SRC, _LIB)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _load(path):
    L = ctypes.CDLL(path)
    vp, u32, i64, f32, i32 = (ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int64,
                              ctypes.c_float, ctypes.c_int)
    L.oracle_mla_rope_rmsnorm_quant.restype = u32
    L.oracle_mla_rope_rmsnorm_quant.argtypes = [
        vp, i32, vp, vp, u32, u32, u32, vp, u32, vp, vp, i64, vp, i32, f32, vp, u32, vp,
        u32, u32, u32, u32, u32, i64, i64, i64, i64, i64, u32, f32, i32]
    L.oracle_mla_rope_rmsnorm_inplace.restype = u32
    L.oracle_mla_rope_rmsnorm_inplace.argtypes = [
        vp, i32, vp, vp, u32, u32, u32, vp, u32, vp, vp, i32, f32, vp, u32, vp, u32, u32, u32,
        i64, i64, i64, u32, f32, i32]
    L.oracle_convert_bf16_to_e4m3.restype = None
    L.oracle_convert_bf16_to_e4m3.argtypes = [vp, vp, i64, f32]
    L.oracle_quantize_rows_e4m3.restype = None
    L.oracle_quantize_rows_e4m3.argtypes = [vp, i64, vp, i64, vp, i64, i64]
    L.oracle_mla_gather_latent.restype = u32
    L.oracle_mla_gather_latent.argtypes = [
        vp, i32, f32, vp, i32, f32, vp, u32, u32, u32, u32, i64, i64, i64, u32, vp, u32, u32]
    L.oracle_mla_gather_latent_dynamic.restype = u32
    L.oracle_mla_gather_latent_dynamic.argtypes = [
        vp, vp, vp, i32, f32, vp, u32, u32, u32, u32, i64, i64, i64, u32, vp, u32, u32]
    L.oracle_qk_rope_paged_ragged.restype = u32
    L.oracle_qk_rope_paged_ragged.argtypes = [
        vp, vp, u32, u32, u32, vp, i32, f32, vp, u32, vp, u32, u32, u32, u32, u32, i64, i64,
        i64, i64, i64, vp, u32, vp, i32, vp, u32, vp, i32]
    L.oracle_rms_norm_kv_cache_paged.restype = u32
    L.oracle_rms_norm_kv_cache_paged.argtypes = [
        vp, vp, u32, vp, u32, u32, u32, u32, u32, i64, i64, i64, i64, i64, vp, u32, f32,
        f32, u32, u32, vp, u32, i32, i32, i32]
    for n in ("oracle_bf16_encode", "oracle_bf16_decode", "oracle_e4m3_encode",
              "oracle_e4m3_decode"):
        getattr(L, n).restype = None
        getattr(L, n).argtypes = [vp, vp, i64]
    L.oracle_rope_pairs_f32.restype = None
    L.oracle_rope_pairs_f32.argtypes = [vp, vp, vp, i64]
    L.oracle_rms_inv.restype = f32
    L.oracle_rms_inv.argtypes = [vp, i64, f32]
    L.oracle_rms_norm_f32.restype = None
    L.oracle_rms_norm_f32.argtypes = [vp, vp, i64, f32, vp]
    L.oracle_has_openmp.restype = i32
    L.oracle_has_openmp.argtypes = []
    return L


def lib():
    global _lib
    if _lib is None:
        if _libpath == _LIB:
            build()
        _lib = _load(_libpath)
    return _lib


class Variant:
    """The oracle's functions bound to another compiled copy of its source
    (used by the tests that plant mistakes in the oracle to prove the pins
    catch them)."""

    def __init__(self, libpath):
        import types

        self._L = _load(libpath)
        g = globals()
        for name in ("bf16_encode", "bf16_decode", "e4m3_encode", "e4m3_decode",
                     "rope_pairs_f32", "rms_inv", "rms_norm_f32", "mla_rope_rmsnorm_quant",
                     "qk_rope_paged_ragged", "rms_norm_kv_cache_paged", "has_openmp",
                     "mla_rope_rmsnorm_inplace", "convert_bf16_to_e4m3", "quantize_rows_e4m3",
                     "mla_gather_latent", "mla_gather_latent_dynamic", "_q_out_buffer"):
            fn = g[name]
            setattr(self, name, types.FunctionType(fn.__code__, dict(g, lib=lambda: self._L),
                                                   name, fn.__defaults__, fn.__closure__))
        self.FLAG_PAGE, self.FLAG_POS, self.FLAG_OFFSETS = FLAG_PAGE, FLAG_POS, FLAG_OFFSETS


def has_openmp() -> bool:
    return bool(lib().oracle_has_openmp())


# ----------------------------------------------------------------- codecs

def bf16_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_bf16_encode(_p(x), _p(out), x.size)
    return out


def bf16_decode(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().oracle_bf16_decode(_p(h), _p(out), h.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode(_p(x), _p(out), x.size)
    return out


def e4m3_decode(c) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float32)
    lib().oracle_e4m3_decode(_p(c), _p(out), c.size)
    return out


# ------------------------------------------------------------ math steps

def rope_pairs_f32(x, cs) -> np.ndarray:
    """Rotate pairs (x[2k], x[2k+1]) by (cs[2k], cs[2k+1]) = (cos, sin), fp32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    cs = np.ascontiguousarray(cs, dtype=np.float32)
    assert x.shape == cs.shape and x.size % 2 == 0
    y = np.empty_like(x)
    lib().oracle_rope_pairs_f32(_p(x), _p(cs), _p(y), x.size // 2)
    return y


def rms_inv(x, eps) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return float(lib().oracle_rms_inv(_p(x), x.size, eps))


def rms_norm_f32(x, w, eps) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    y = np.empty_like(x)
    lib().oracle_rms_norm_f32(_p(x), _p(w), x.size, eps, _p(y))
    return y


# ----------------------------------------------------------- entry points

def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _q_out_buffer(q, q_rope_out, out_dtype):
    if q_rope_out is None:
        q_rope_out = np.zeros(q.shape, dtype=np.uint16 if out_dtype == 0 else np.uint8)
    return q_rope_out


def mla_rope_rmsnorm_quant(w, q_rope_out=None, cache_data=None, nthreads=1, T=None,
                           kv_row_stride=None, kv_in=None, out_dtype=0):
    """Run the MLA write on workload ``w``.

    Returns ``(q_rope_out, cache_data, flags)``.  ``cache_data`` defaults to a
    copy of ``w.cache.data`` and ``q_rope_out`` to zeros (bf16 bits, or E4M3
    codes with ``out_dtype`` 1); both are modified in place when given.
    """
    c = w.cache
    T = w.T if T is None else T
    q = _c(w.q_rope, np.uint16)
    q_rope_out = _q_out_buffer(q, q_rope_out, out_dtype)
    if cache_data is None:
        cache_data = c.data.copy()
    kv = _c(w.kv_in if kv_in is None else kv_in, np.uint16)
    stride = kv.shape[-1] if kv_row_stride is None else kv_row_stride
    off = _c(w.offsets, np.uint32)
    fr = _c(w.freqs, np.float32)
    g = _c(w.gamma, np.uint16)
    s = c.strides
    flags = lib().oracle_mla_rope_rmsnorm_quant(
        _p(q_rope_out), out_dtype, _p(q), _p(off), len(off) - 1, T,
        q.shape[1] if q.ndim == 3 else 0, _p(fr), fr.shape[0], _p(g), _p(kv), stride,
        _p(cache_data), c.dtype, c.scale, _p(c.page_table), c.max_pages_per_seq,
        _p(c.cache_lengths), c.num_pages, c.num_layers, c.page_size, c.num_heads, c.head_size,
        s[0], s[1], s[2], s[3], s[4], w.layer_idx, w.epsilon, nthreads)
    return q_rope_out, cache_data, int(flags)


def mla_rope_rmsnorm_inplace(w, q_rope_out=None, cache_data=None, nthreads=1, out_dtype=0):
    """In-place variant: the new latent rows are read from ``w.cache`` (place
    them with ``workloads.place_latent_rows``).  Returns (q_out, cache, flags)."""
    c = w.cache
    q = _c(w.q_rope, np.uint16)
    q_rope_out = _q_out_buffer(q, q_rope_out, out_dtype)
    if cache_data is None:
        cache_data = c.data.copy()
    off = _c(w.offsets, np.uint32)
    fr = _c(w.freqs, np.float32)
    g = _c(w.gamma, np.uint16)
    s = c.strides
    flags = lib().oracle_mla_rope_rmsnorm_inplace(
        _p(q_rope_out), out_dtype, _p(q), _p(off), len(off) - 1, w.T,
        q.shape[1] if q.ndim == 3 else 0, _p(fr), fr.shape[0], _p(g), _p(cache_data), c.dtype,
        c.scale, _p(c.page_table), c.max_pages_per_seq, _p(c.cache_lengths), c.num_pages,
        c.num_layers, c.page_size, s[0], s[2], s[3], w.layer_idx, w.epsilon, nthreads)
    return q_rope_out, cache_data, int(flags)


def convert_bf16_to_e4m3(x_bits, scale=1.0) -> np.ndarray:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_convert_bf16_to_e4m3(_p(x), _p(out), x.size, scale)
    return out


def quantize_rows_e4m3(x_bits):
    """Per-row dynamic FP8: returns (codes uint8 [rows, cols], scales f32 [rows])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    out = np.empty(x.shape, dtype=np.uint8)
    sc = np.empty(rows, dtype=np.float32)
    lib().oracle_quantize_rows_e4m3(_p(x), cols, _p(out), cols, _p(sc), rows, cols)
    return out, sc


def mla_gather_latent(cache, layer_idx, ctx_offsets, out_dtype=0, out_scale=1.0, out=None):
    """Paged -> contiguous latent rows; returns (out [rows, 576], flags)."""
    off = np.ascontiguousarray(ctx_offsets, dtype=np.uint32)
    rows = int(off[-1]) if off.size else 0
    if out is None:
        out = np.zeros((rows, 576), dtype=np.uint16 if out_dtype == 0 else np.uint8)
    s = cache.strides
    flags = lib().oracle_mla_gather_latent(
        _p(out), out_dtype, out_scale, _p(cache.data), cache.dtype, cache.scale,
        _p(cache.page_table), cache.max_pages_per_seq, cache.num_pages, cache.num_layers,
        cache.page_size, s[0], s[2], s[3], layer_idx, _p(off), len(off) - 1, rows)
    return out, int(flags)


def mla_gather_latent_dynamic(cache, layer_idx, ctx_offsets, out=None, scales=None):
    """Paged -> contiguous latent rows with per-row dynamic FP8; returns
    (codes uint8 [rows, 576], scales f32 [rows], flags)."""
    off = np.ascontiguousarray(ctx_offsets, dtype=np.uint32)
    rows = int(off[-1]) if off.size else 0
    if out is None:
        out = np.zeros((rows, 576), dtype=np.uint8)
    if scales is None:
        scales = np.zeros(rows, dtype=np.float32)
    s = cache.strides
    flags = lib().oracle_mla_gather_latent_dynamic(
        _p(out), _p(scales), _p(cache.data), cache.dtype, cache.scale, _p(cache.page_table),
        cache.max_pages_per_seq, cache.num_pages, cache.num_layers, cache.page_size, s[0], s[2],
        s[3], layer_idx, _p(off), len(off) - 1, rows)
    return out, scales, int(flags)


def qk_rope_paged_ragged(w, output=None, cache_data=None, nthreads=1, T=None):
    """Run the GQA Q/K rotation on workload ``w``; returns (output, cache, flags)."""
    c = w.cache
    T = w.T if T is None else T
    q = _c(w.q_proj, np.uint16)
    if output is None:
        output = np.zeros(q.shape, dtype=np.uint16)
    if cache_data is None:
        cache_data = c.data.copy()
    off = _c(w.offsets, np.uint32)
    fr = _c(w.freqs, np.float32)
    pid = None if w.position_ids is None else _c(w.position_ids, np.uint32)
    sec = None if w.mrope_section is None else _c(w.mrope_section, np.uint32)
    s = c.strides
    flags = lib().oracle_qk_rope_paged_ragged(
        _p(q), _p(off), len(off) - 1, T, q.shape[1], _p(cache_data), c.dtype, c.scale,
        _p(c.page_table),
        c.max_pages_per_seq, _p(c.cache_lengths), c.num_pages, c.num_layers, c.page_size,
        c.num_heads, c.head_size, s[0], s[1], s[2], s[3], s[4], _p(fr), fr.shape[0],
        _p(pid), int(w.interleaved), _p(sec), w.layer_idx, _p(output), nthreads)
    return output, cache_data, int(flags)


def rms_norm_kv_cache_paged(w, cache_data=None, nthreads=1, per_head_norm=None, T=None):
    """Run the in-place K-cache RMSNorm on workload ``w``; returns (cache, flags)."""
    if per_head_norm is None:
        per_head_norm = getattr(w, "per_head_norm", True)
    c = w.cache
    T = w.T if T is None else T
    if cache_data is None:
        cache_data = c.data.copy()
    off = _c(w.offsets, np.uint32)
    g = _c(w.gamma, np.uint16)
    s = c.strides
    flags = lib().oracle_rms_norm_kv_cache_paged(
        _p(cache_data), _p(c.page_table), c.max_pages_per_seq, _p(c.cache_lengths),
        c.num_pages, c.num_layers, c.page_size, c.num_heads, c.head_size, s[0], s[1], s[2],
        s[3], s[4], _p(g), g.size, w.epsilon, w.weight_offset, w.layer_idx, T, _p(off),
        len(off) - 1, int(w.multiply_before_cast), int(per_head_norm), nthreads)
    return cache_data, int(flags)
