"""The C ABI library loads, exports what include/kvw.h declares, and rejects
bad host arguments before touching the GPU (these calls return before any
CUDA call, so they run without a device)."""
import ctypes
import re
import subprocess

import pytest

from gqa_kv_cache_mla_gb300 import kvw

FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced
ODD = 0x10008   # an 8-byte but not 16-byte aligned address


def test_exports_every_header_function():
    names = kvw.header_functions()
    assert set(names) == {"kvw_mla_rope_rmsnorm_quant", "kvw_mla_rope_rmsnorm_inplace",
                          "kvw_qk_rope_paged_ragged", "kvw_rms_norm_kv_cache_paged",
                          "kvw_mla_gather_latent", "kvw_mla_gather_latent_fp8_dynamic",
                          "kvw_convert_bf16_to_fp8_e4m3",
                          "kvw_quantize_fp8_rows", "kvw_status_string", "kvw_version"}
    for n in names:
        assert hasattr(kvw.lib, n)
    out = subprocess.run(["nm", "-D", "--defined-only", kvw.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (kvw_\w+)", out))
    # exactly the header's functions: test hooks live in a separate test build only
    assert exported == set(names)


def test_status_strings_and_version():
    assert kvw.version() == 110
    assert kvw.status_string(0) == "KVW_OK"
    for s in (1, 2, 3):
        assert kvw.status_string(s).startswith("KVW_E")
    assert "unknown" in kvw.status_string(99)


def test_struct_layout_matches_header():
    # 8 (data) + 4 + 4 + 8 + 4 (+4 pad) + 8 + 5*4 (+4 pad) + 5*8
    assert ctypes.sizeof(kvw.PagedCacheT) == 104
    assert kvw.PagedCacheT.stride_page.offset == 64


def _mla_cache(**kw):
    d = dict(data=FAKE, dtype=kvw.DTYPE_FP8_E4M3, page_table=FAKE, cache_lengths=FAKE,
             num_pages=8, num_layers=2, page_size=16, num_heads=1, head_size=576,
             strides=(2 * 16 * 576, 0, 16 * 576, 576, 576), max_pages_per_seq=4)
    d.update(kw)
    return kvw.paged_cache(**d)


def _mla(cache, **kw):
    a = dict(q_rope_out=FAKE, out_dtype=kvw.DTYPE_BF16, q_rope=FAKE, offsets=FAKE, B=2, T=8, H=4,
             freqs=FAKE, freq_dtype=kvw.DTYPE_F32, rows=64, gamma=FAKE,
             gamma_dtype=kvw.DTYPE_BF16, kv=FAKE, stride=576, layer=1, eps=1e-6)
    a.update(kw)
    return kvw.lib.kvw_mla_rope_rmsnorm_quant(
        a["q_rope_out"], a["out_dtype"], a["q_rope"], a["offsets"], a["B"], a["T"], a["H"],
        a["freqs"], a["freq_dtype"], a["rows"], a["gamma"], a["gamma_dtype"], a["kv"], a["stride"],
        None if cache is None else ctypes.byref(cache), a["layer"], a["eps"], None, 0)


@pytest.mark.parametrize("cache_kw,call_kw,want", [
    ({}, {"T": 0}, kvw.KVW_OK),  # nothing to do: no launch
    ({}, {"out_dtype": kvw.DTYPE_F32}, kvw.KVW_EUNSUPPORTED),
    ({}, {"freq_dtype": kvw.DTYPE_BF16}, kvw.KVW_EUNSUPPORTED),
    ({"head_size": 512}, {}, kvw.KVW_EUNSUPPORTED),
    ({"num_heads": 2}, {}, kvw.KVW_EUNSUPPORTED),
    ({"dtype": kvw.DTYPE_F32}, {}, kvw.KVW_EUNSUPPORTED),
    ({}, {"B": 8193}, kvw.KVW_EUNSUPPORTED),
    ({}, {"stride": 570}, kvw.KVW_EINVAL),
    ({}, {"stride": 580}, kvw.KVW_EINVAL),
    ({}, {"layer": 2}, kvw.KVW_EINVAL),
    ({}, {"kv": ODD}, kvw.KVW_EINVAL),
    ({}, {"q_rope_out": ODD}, kvw.KVW_EINVAL),
    ({}, {"q_rope": None}, kvw.KVW_EINVAL),
    ({}, {"offsets": None}, kvw.KVW_EINVAL),
    ({}, {"rows": 0}, kvw.KVW_EINVAL),
    ({}, {"eps": -1.0}, kvw.KVW_EINVAL),
    ({"data": ODD}, {}, kvw.KVW_EINVAL),
    ({"page_size": 0}, {}, kvw.KVW_EINVAL),
    ({"strides": (2 * 16 * 576, 0, 16 * 576, 570, 576)}, {}, kvw.KVW_EINVAL),
])
def test_mla_host_argument_checks(cache_kw, call_kw, want):
    assert _mla(_mla_cache(**cache_kw), **call_kw) == want


def test_mla_null_cache():
    assert _mla(None) == kvw.KVW_EINVAL


def _gqa_cache(**kw):
    d = dict(data=FAKE, dtype=kvw.DTYPE_BF16, page_table=FAKE, cache_lengths=FAKE, num_pages=8,
             num_layers=2, page_size=16, num_heads=8, head_size=128,
             strides=(2 * 2 * 16 * 8 * 128, 2 * 16 * 8 * 128, 16 * 8 * 128, 8 * 128, 128),
             max_pages_per_seq=4)
    d.update(kw)
    return kvw.paged_cache(**d)


def _gqa(cache, T=8, Hq=32, pos=FAKE, sec=None, out=FAKE, layer=1):
    s = None if sec is None else ctypes.cast((ctypes.c_uint32 * 3)(*sec), ctypes.c_void_p)
    return kvw.lib.kvw_qk_rope_paged_ragged(FAKE, FAKE, 2, T, Hq, ctypes.byref(cache), FAKE, 64,
                                           pos, 1, s, layer, out, None, 0)


@pytest.mark.parametrize("cache_kw,call_kw,want", [
    ({}, {"T": 0}, kvw.KVW_OK),
    ({"head_size": 72}, {}, kvw.KVW_EUNSUPPORTED),
    ({"head_size": 1024}, {}, kvw.KVW_EUNSUPPORTED),
    ({"dtype": kvw.DTYPE_F32}, {}, kvw.KVW_EUNSUPPORTED),
    ({"dtype": kvw.DTYPE_FP8_E4M3, "scale": 0.0}, {}, kvw.KVW_EINVAL),
    ({"dtype": kvw.DTYPE_FP8_E4M3, "strides": (2 * 2 * 16 * 8 * 128, 2 * 16 * 8 * 128,
                                               16 * 8 * 128, 8 * 128, 136)}, {}, kvw.KVW_EINVAL),
    ({}, {"Hq": 200}, kvw.KVW_EUNSUPPORTED),
    ({}, {"sec": (16, 24, 23)}, kvw.KVW_EINVAL),
    ({}, {"sec": (16, 24, 24), "pos": None}, kvw.KVW_EINVAL),
    ({}, {"out": ODD}, kvw.KVW_EINVAL),
    ({}, {"layer": 5}, kvw.KVW_EINVAL),
    ({"strides": (2 * 2 * 16 * 8 * 128, 2 * 16 * 8 * 128, 16 * 8 * 128, 8 * 128, 132)}, {},
     kvw.KVW_EINVAL),
])
def test_gqa_host_argument_checks(cache_kw, call_kw, want):
    assert _gqa(_gqa_cache(**cache_kw), **call_kw) == want


@pytest.mark.parametrize("cache_kw,G,per_head,want", [
    ({}, 129, True, kvw.KVW_EINVAL),
    ({}, 0, True, kvw.KVW_EINVAL),
    ({}, 128, False, kvw.KVW_EINVAL),
    ({}, 1024, False, kvw.KVW_OK),  # T = 0 below: valid, nothing launched
    ({"dtype": kvw.DTYPE_FP8_E4M3}, 128, True, kvw.KVW_EUNSUPPORTED),
    ({"head_size": 4096}, 4096, True, kvw.KVW_EUNSUPPORTED),
])
def test_knorm_host_argument_checks(cache_kw, G, per_head, want):
    c = _gqa_cache(**cache_kw)
    T = 0 if want == kvw.KVW_OK else 8
    st = kvw.lib.kvw_rms_norm_kv_cache_paged(ctypes.byref(c), FAKE, G, 1e-6, 0.0, 1, T, FAKE, 2,
                                             1, int(per_head), None, 0)
    assert st == want


def test_binding_raises_on_error_status():
    with pytest.raises(kvw.KvwError):
        kvw._done(kvw.KVW_EINVAL, "x", True)
    assert kvw._done(kvw.KVW_EINVAL, "x", False) == kvw.KVW_EINVAL



def test_inplace_host_checks():
    c = _mla_cache()
    f = kvw.lib.kvw_mla_rope_rmsnorm_inplace
    args = [FAKE, kvw.DTYPE_BF16, FAKE, FAKE, 2, 8, 4, FAKE, kvw.DTYPE_F32, 64, FAKE,
            kvw.DTYPE_BF16, ctypes.byref(c), 1, 1e-6, None, 0]
    assert f(*args[:12], None, *args[13:]) == kvw.KVW_EINVAL  # no cache
    a = list(args)
    a[5] = 0
    assert f(*a) == kvw.KVW_OK  # no tokens
    a = list(args)
    a[0] = ODD
    assert f(*a) == kvw.KVW_EINVAL
    c2 = _mla_cache(scale=-1.0)
    a = list(args)
    a[12] = ctypes.byref(c2)
    assert f(*a) == kvw.KVW_EINVAL


def test_gather_host_checks():
    c = _mla_cache()
    f = kvw.lib.kvw_mla_gather_latent
    assert f(FAKE, kvw.DTYPE_BF16, 1.0, ctypes.byref(c), 1, FAKE, 2, 0, None, 0) == kvw.KVW_OK
    assert f(FAKE, kvw.DTYPE_F32, 1.0, ctypes.byref(c), 1, FAKE, 2, 8, None, 0) == \
        kvw.KVW_EUNSUPPORTED
    assert f(ODD, kvw.DTYPE_BF16, 1.0, ctypes.byref(c), 1, FAKE, 2, 8, None, 0) == kvw.KVW_EINVAL
    assert f(FAKE, kvw.DTYPE_FP8_E4M3, 0.0, ctypes.byref(c), 1, FAKE, 2, 8, None, 0) == \
        kvw.KVW_EINVAL
    assert f(FAKE, kvw.DTYPE_BF16, 1.0, ctypes.byref(c), 2, FAKE, 2, 8, None, 0) == kvw.KVW_EINVAL
    c2 = _mla_cache(head_size=512)
    assert f(FAKE, kvw.DTYPE_BF16, 1.0, ctypes.byref(c2), 1, FAKE, 2, 8, None, 0) == \
        kvw.KVW_EUNSUPPORTED


def test_codec_host_checks():
    conv = kvw.lib.kvw_convert_bf16_to_fp8_e4m3
    assert conv(FAKE, FAKE, 0, 1.0, 0) == kvw.KVW_OK
    assert conv(FAKE, FAKE, 12, 1.0, 0) == kvw.KVW_EINVAL  # not a multiple of 8
    assert conv(FAKE, ODD, 16, 1.0, 0) == kvw.KVW_EINVAL
    assert conv(FAKE, FAKE, 16, 0.0, 0) == kvw.KVW_EINVAL
    q = kvw.lib.kvw_quantize_fp8_rows
    assert q(FAKE, FAKE, FAKE, 0, 64, 64, 64, 0) == kvw.KVW_OK
    assert q(FAKE, FAKE, FAKE, 4, 60, 64, 64, 0) == kvw.KVW_EINVAL
    assert q(FAKE, FAKE, FAKE, 4, 64, 60, 64, 0) == kvw.KVW_EINVAL
    assert q(FAKE, FAKE, ODD, 4, 64, 64, 64, 0) == kvw.KVW_EINVAL


def test_binding_output_type_follows_the_buffer():
    """The binding derives the q / gather output type from the output tensor and
    rejects a type wider than the buffer (the kernel would write past it)."""
    import torch

    u8 = torch.zeros(16, dtype=torch.uint8)
    i16 = torch.zeros(16, dtype=torch.int16)
    assert kvw._out_dtype(u8, None, "x") == kvw.DTYPE_FP8_E4M3
    assert kvw._out_dtype(i16, None, "x") == kvw.DTYPE_BF16
    assert kvw._out_dtype(i16, kvw.DTYPE_BF16, "x") == kvw.DTYPE_BF16
    with pytest.raises(ValueError):
        kvw._out_dtype(u8, kvw.DTYPE_BF16, "x")
    with pytest.raises(ValueError):
        kvw._out_dtype(i16, kvw.DTYPE_FP8_E4M3, "x")


def test_gather_dynamic_host_checks():
    c = _mla_cache()
    f = kvw.lib.kvw_mla_gather_latent_fp8_dynamic
    assert f(FAKE, FAKE, ctypes.byref(c), 1, FAKE, 2, 0, None, 0) == kvw.KVW_OK
    assert f(ODD, FAKE, ctypes.byref(c), 1, FAKE, 2, 8, None, 0) == kvw.KVW_EINVAL
    assert f(FAKE, FAKE + 2, ctypes.byref(c), 1, FAKE, 2, 8, None, 0) == kvw.KVW_EINVAL
    assert f(FAKE, None, ctypes.byref(c), 1, FAKE, 2, 8, None, 0) == kvw.KVW_EINVAL
    assert f(FAKE, FAKE, ctypes.byref(c), 2, FAKE, 2, 8, None, 0) == kvw.KVW_EINVAL
    assert f(FAKE, FAKE, None, 1, FAKE, 2, 8, None, 0) == kvw.KVW_EINVAL
    c2 = _mla_cache(head_size=512)
    assert f(FAKE, FAKE, ctypes.byref(c2), 1, FAKE, 2, 8, None, 0) == kvw.KVW_EUNSUPPORTED


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library the binding raises: there is no fallback path
    that could compute anything elsewhere."""
    monkeypatch.setattr(kvw, "LIB_PATH", str(tmp_path / "libkvw.so"))
    with pytest.raises(ImportError, match="library missing"):
        kvw._load()


def test_product_package_does_not_import_the_oracle():
    """The package (binding, device helpers, generators, profiling driver)
    never imports the CPU reference: only tests and the benchmark's baseline
    leg may."""
    import pathlib

    pkg = pathlib.Path(kvw.__file__).parent
    for f in pkg.glob("*.py"):
        text = f.read_text()
        assert "import oracle" not in text and "from oracle" not in text, f.name
