"""Python binding of the kvw C ABI (``include/kvw.h``).

Argument marshalling only: every function forwards device pointers, sizes
and the current CUDA stream to the function of the same name in
``libkvw.so`` and returns its status (raising :class:`KvwError` on a
non-zero status unless ``check=False``).  All computation happens in the
library's sm_103a kernels; there is no other code path.  The library is
built in-tree by ``python -m gqa_kv_cache_mla_gb300.build``; importing this
module without it raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvw.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kvw.h")

KVW_OK, KVW_EINVAL, KVW_EUNSUPPORTED, KVW_ECUDA = 0, 1, 2, 3
DTYPE_BF16, DTYPE_FP8_E4M3, DTYPE_F32 = 0, 1, 2
ERR_PAGE, ERR_POSITION, ERR_OFFSETS = 1, 2, 4
PAGE_UNMAPPED = 0xFFFFFFFF


class KvwError(RuntimeError):
    def __init__(self, status, where):
        super().__init__("%s returned %d (%s)" % (where, status, status_string(status)))
        self.status = status


class PagedCacheT(ctypes.Structure):
    """Mirror of ``kvw_paged_cache_t``."""

    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("page_table", ctypes.c_void_p),
        ("max_pages_per_seq", ctypes.c_uint32),
        ("cache_lengths", ctypes.c_void_p),
        ("num_pages", ctypes.c_uint32),
        ("num_layers", ctypes.c_uint32),
        ("page_size", ctypes.c_uint32),
        ("num_heads", ctypes.c_uint32),
        ("head_size", ctypes.c_uint32),
        ("stride_page", ctypes.c_int64),
        ("stride_kv", ctypes.c_int64),
        ("stride_layer", ctypes.c_int64),
        ("stride_token", ctypes.c_int64),
        ("stride_head", ctypes.c_int64),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("kvw CUDA library missing (%s): build it with "
                          "`python -m gqa_kv_cache_mla_gb300.build`" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, u32, i32, i64, f32 = (ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int32, ctypes.c_int64,
                              ctypes.c_float)
    pc = ctypes.POINTER(PagedCacheT)
    L.kvw_mla_rope_rmsnorm_quant.restype = ctypes.c_int
    L.kvw_mla_rope_rmsnorm_quant.argtypes = [vp, i32, vp, vp, u32, u32, u32, vp, i32, u32, vp, i32,
                                             vp, i64, pc, u32, f32, vp, vp]
    L.kvw_qk_rope_paged_ragged.restype = ctypes.c_int
    L.kvw_qk_rope_paged_ragged.argtypes = [vp, vp, u32, u32, u32, pc, vp, u32, vp, ctypes.c_int,
                                           vp, u32, vp, vp, vp]
    L.kvw_rms_norm_kv_cache_paged.restype = ctypes.c_int
    L.kvw_rms_norm_kv_cache_paged.argtypes = [pc, vp, u32, f32, f32, u32, u32, vp, u32,
                                              ctypes.c_int, ctypes.c_int, vp, vp]
    L.kvw_mla_rope_rmsnorm_inplace.restype = ctypes.c_int
    L.kvw_mla_rope_rmsnorm_inplace.argtypes = [vp, i32, vp, vp, u32, u32, u32, vp, i32, u32, vp,
                                               i32, pc, u32, f32, vp, vp]
    L.kvw_mla_gather_latent.restype = ctypes.c_int
    L.kvw_mla_gather_latent.argtypes = [vp, i32, f32, pc, u32, vp, u32, u32, vp, vp]
    L.kvw_mla_gather_latent_fp8_dynamic.restype = ctypes.c_int
    L.kvw_mla_gather_latent_fp8_dynamic.argtypes = [vp, vp, pc, u32, vp, u32, u32, vp, vp]
    L.kvw_convert_bf16_to_fp8_e4m3.restype = ctypes.c_int
    L.kvw_convert_bf16_to_fp8_e4m3.argtypes = [vp, vp, ctypes.c_uint64, f32, vp]
    L.kvw_quantize_fp8_rows.restype = ctypes.c_int
    L.kvw_quantize_fp8_rows.argtypes = [vp, vp, vp, u32, u32, i64, i64, vp]
    L.kvw_status_string.restype = ctypes.c_char_p
    L.kvw_status_string.argtypes = [ctypes.c_int]
    L.kvw_version.restype = ctypes.c_int
    L.kvw_version.argtypes = []
    return L


lib = _load()


def header_functions():
    """Names of the functions ``include/kvw.h`` declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(kvw_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return lib.kvw_status_string(status).decode()


def version() -> int:
    return lib.kvw_version()


def _ptr(x):
    """Device address of a tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _done(status, name, check):
    if check and status != KVW_OK:
        raise KvwError(status, name)
    return status


def paged_cache(data, dtype, page_table, cache_lengths, num_pages, num_layers, page_size,
                num_heads, head_size, strides, scale=1.0, max_pages_per_seq=None) -> PagedCacheT:
    """Fill a ``kvw_paged_cache_t``; ``strides`` = (page, kv, layer, token, head) in elements."""
    if max_pages_per_seq is None:
        max_pages_per_seq = page_table.shape[-1]
    s = PagedCacheT()
    s.data = _ptr(data)
    s.dtype = dtype
    s.scale = scale
    s.page_table = _ptr(page_table)
    s.max_pages_per_seq = max_pages_per_seq
    s.cache_lengths = _ptr(cache_lengths)
    s.num_pages, s.num_layers, s.page_size = num_pages, num_layers, page_size
    s.num_heads, s.head_size = num_heads, head_size
    (s.stride_page, s.stride_kv, s.stride_layer, s.stride_token, s.stride_head) = strides
    return s


def _out_dtype(out, out_dtype, name):
    """The element type code of an output buffer: taken from the tensor's
    element size when not given (1 byte: FP8 E4M3, 2 bytes: bf16), and
    checked against it when given, so the kernel never writes a wider type
    into a narrower buffer."""
    size = out.element_size() if hasattr(out, "element_size") else None
    if out_dtype is None:
        if size not in (1, 2):
            raise ValueError("%s: give out_dtype for an output without an element size" % name)
        return DTYPE_FP8_E4M3 if size == 1 else DTYPE_BF16
    want = {DTYPE_FP8_E4M3: 1, DTYPE_BF16: 2}.get(out_dtype)
    if size is not None and want is not None and size != want:
        raise ValueError("%s: out_dtype %d needs %d-byte elements, the output has %d" % (
            name, out_dtype, want, size))
    return out_dtype


def kvw_mla_rope_rmsnorm_quant(q_rope_out, q_rope, input_row_offsets, freqs_cis, gamma, kv_in,
                               cache: PagedCacheT, layer_idx: int, epsilon: float, err_flags=None,
                               stream=None, *, num_batches=None, tot_seq_len=None,
                               num_heads=None, freqs_rows=None, kv_row_stride=None,
                               out_dtype=None, freq_dtype=DTYPE_F32,
                               gamma_dtype=DTYPE_BF16, check=True) -> int:
    out_dtype = _out_dtype(q_rope_out, out_dtype, "kvw_mla_rope_rmsnorm_quant")
    B = input_row_offsets.shape[0] - 1 if num_batches is None else num_batches
    T = q_rope.shape[0] if tot_seq_len is None else tot_seq_len
    H = q_rope.shape[1] if num_heads is None else num_heads
    rows = freqs_cis.shape[0] if freqs_rows is None else freqs_rows
    stride = kv_in.stride(0) if kv_row_stride is None else kv_row_stride
    st = lib.kvw_mla_rope_rmsnorm_quant(
        _ptr(q_rope_out), out_dtype, _ptr(q_rope), _ptr(input_row_offsets), B, T, H,
        _ptr(freqs_cis), freq_dtype, rows, _ptr(gamma), gamma_dtype, _ptr(kv_in), stride,
        ctypes.byref(cache), layer_idx, epsilon, _ptr(err_flags), _stream(stream))
    return _done(st, "kvw_mla_rope_rmsnorm_quant", check)


def kvw_mla_rope_rmsnorm_inplace(q_rope_out, q_rope, input_row_offsets, freqs_cis, gamma,
                                 cache: PagedCacheT, layer_idx: int, epsilon: float,
                                 err_flags=None, stream=None, *, num_batches=None,
                                 tot_seq_len=None, num_heads=None, freqs_rows=None,
                                 out_dtype=None, freq_dtype=DTYPE_F32,
                                 gamma_dtype=DTYPE_BF16, check=True) -> int:
    out_dtype = _out_dtype(q_rope_out, out_dtype, "kvw_mla_rope_rmsnorm_inplace")
    B = input_row_offsets.shape[0] - 1 if num_batches is None else num_batches
    T = q_rope.shape[0] if tot_seq_len is None else tot_seq_len
    H = q_rope.shape[1] if num_heads is None else num_heads
    rows = freqs_cis.shape[0] if freqs_rows is None else freqs_rows
    st = lib.kvw_mla_rope_rmsnorm_inplace(
        _ptr(q_rope_out), out_dtype, _ptr(q_rope), _ptr(input_row_offsets), B, T, H,
        _ptr(freqs_cis), freq_dtype, rows, _ptr(gamma), gamma_dtype, ctypes.byref(cache),
        layer_idx, epsilon, _ptr(err_flags), _stream(stream))
    return _done(st, "kvw_mla_rope_rmsnorm_inplace", check)


def kvw_mla_gather_latent(out, out_dtype: int, out_scale: float, cache: PagedCacheT,
                          layer_idx: int, ctx_offsets, err_flags=None, stream=None, *,
                          num_batches=None, total_rows=None, check=True) -> int:
    out_dtype = _out_dtype(out, out_dtype, "kvw_mla_gather_latent")
    B = ctx_offsets.shape[0] - 1 if num_batches is None else num_batches
    rows = out.shape[0] if total_rows is None else total_rows
    st = lib.kvw_mla_gather_latent(_ptr(out), out_dtype, out_scale, ctypes.byref(cache),
                                   layer_idx, _ptr(ctx_offsets), B, rows, _ptr(err_flags),
                                   _stream(stream))
    return _done(st, "kvw_mla_gather_latent", check)


def kvw_mla_gather_latent_fp8_dynamic(out_codes, out_scales, cache: PagedCacheT, layer_idx: int,
                                      ctx_offsets, err_flags=None, stream=None, *,
                                      num_batches=None, total_rows=None, check=True) -> int:
    B = ctx_offsets.shape[0] - 1 if num_batches is None else num_batches
    rows = out_codes.shape[0] if total_rows is None else total_rows
    st = lib.kvw_mla_gather_latent_fp8_dynamic(_ptr(out_codes), _ptr(out_scales),
                                               ctypes.byref(cache), layer_idx, _ptr(ctx_offsets),
                                               B, rows, _ptr(err_flags), _stream(stream))
    return _done(st, "kvw_mla_gather_latent_fp8_dynamic", check)


def kvw_convert_bf16_to_fp8_e4m3(out, inp, scale: float = 1.0, stream=None, *, n=None,
                                 check=True) -> int:
    n = inp.numel() if n is None else n
    st = lib.kvw_convert_bf16_to_fp8_e4m3(_ptr(out), _ptr(inp), n, scale, _stream(stream))
    return _done(st, "kvw_convert_bf16_to_fp8_e4m3", check)


def kvw_quantize_fp8_rows(out_codes, out_scales, inp, stream=None, *, rows=None, cols=None,
                          in_row_stride=None, out_row_stride=None, check=True) -> int:
    rows = inp.shape[0] if rows is None else rows
    cols = inp.shape[1] if cols is None else cols
    ins = inp.stride(0) if in_row_stride is None else in_row_stride
    outs = out_codes.stride(0) if out_row_stride is None else out_row_stride
    st = lib.kvw_quantize_fp8_rows(_ptr(out_codes), _ptr(out_scales), _ptr(inp), rows, cols, ins,
                                   outs, _stream(stream))
    return _done(st, "kvw_quantize_fp8_rows", check)


def kvw_qk_rope_paged_ragged(q_proj, input_row_offsets, cache: PagedCacheT, freqs_cis,
                             position_ids, interleaved: bool, mrope_section, layer_idx: int,
                             output, err_flags=None, stream=None, *, num_batches=None,
                             tot_seq_len=None, num_q_heads=None, freqs_rows=None,
                             check=True) -> int:
    B = input_row_offsets.shape[0] - 1 if num_batches is None else num_batches
    T = q_proj.shape[0] if tot_seq_len is None else tot_seq_len
    Hq = q_proj.shape[1] if num_q_heads is None else num_q_heads
    rows = freqs_cis.shape[0] if freqs_rows is None else freqs_rows
    sec = None
    if mrope_section is not None:
        sec = (ctypes.c_uint32 * 3)(*[int(v) for v in mrope_section])
    st = lib.kvw_qk_rope_paged_ragged(
        _ptr(q_proj), _ptr(input_row_offsets), B, T, Hq, ctypes.byref(cache), _ptr(freqs_cis),
        rows, _ptr(position_ids), int(bool(interleaved)),
        ctypes.cast(sec, ctypes.c_void_p) if sec is not None else None, layer_idx, _ptr(output),
        _ptr(err_flags), _stream(stream))
    return _done(st, "kvw_qk_rope_paged_ragged", check)


def kvw_rms_norm_kv_cache_paged(cache: PagedCacheT, gamma, epsilon: float, weight_offset: float,
                                layer_idx: int, total_seq_len: int, input_row_offsets,
                                multiply_before_cast: bool = True, per_head_norm: bool = True,
                                err_flags=None, stream=None, *, gamma_len=None,
                                num_batches=None, check=True) -> int:
    G = gamma.shape[0] if gamma_len is None else gamma_len
    B = input_row_offsets.shape[0] - 1 if num_batches is None else num_batches
    st = lib.kvw_rms_norm_kv_cache_paged(
        ctypes.byref(cache), _ptr(gamma), G, epsilon, weight_offset, layer_idx, total_seq_len,
        _ptr(input_row_offsets), B, int(bool(multiply_before_cast)), int(bool(per_head_norm)),
        _ptr(err_flags), _stream(stream))
    return _done(st, "kvw_rms_norm_kv_cache_paged", check)
