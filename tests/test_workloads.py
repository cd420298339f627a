"""The seeded input generators are deterministic: the same seed gives the same
bytes (the GPU path and the oracle read the same inputs, and a failing case
can be rebuilt from its seed), and another seed gives other bytes."""
import dataclasses

import numpy as np
import pytest

from gqa_kv_cache_mla_gb300 import workloads as W


def _arrays(obj, prefix=""):
    """Every numpy array reachable from a workload (dataclasses, nested)."""
    out = {}
    for f in dataclasses.fields(obj):
        v = getattr(obj, f.name)
        if isinstance(v, np.ndarray):
            out[prefix + f.name] = v
        elif dataclasses.is_dataclass(v):
            out.update(_arrays(v, prefix + f.name + "."))
    return out


BUILDERS = {
    "mla_tiny": lambda s: W.mla_tiny(W.DTYPE_FP8_E4M3, seed=s),
    "mla_small": lambda s: W.mla_workload("m", s, [3, 0, 9], [5, 40, 0], num_heads=3,
                                          page_size=16, max_seq_len=64,
                                          cache_dtype=W.DTYPE_BF16, outlier_frac=0.05),
    "mla_inplace": lambda s: W.mla_inplace(W.mla_tiny(W.DTYPE_BF16, seed=s)),
    "gather": lambda s: W.mla_gather(W.mla_tiny(W.DTYPE_BF16, seed=s), seed=s + 1),
    "gqa_mrope": lambda s: W.gqa_workload("g", s, [3, 5, 1], [0, 7, 30], 4, 2, 32,
                                          page_size=16, freqs_rows=64, base=10000.0,
                                          interleaved=False, position_mode="mrope",
                                          mrope_section=(4, 6, 6)),
    "gqa_fp8": lambda s: W.gqa_workload("g", s, [3, 5], [0, 7], 2, 2, 32, page_size=16,
                                        freqs_rows=64, base=10000.0, interleaved=True,
                                        cache_dtype=W.DTYPE_FP8_E4M3, scale=0.5),
    "knorm": lambda s: W.knorm_workload("k", s, [2, 9], [5, 0], 3, 32, page_size=8,
                                        gamma_len=24, weight_offset=0.5),
    "codec_rows": lambda s: W.fp8_quant_rows(rows=16, cols=64, seed=s),
    "codec_flat": lambda s: W.fp8_convert(n=1024, seed=s),
}


@pytest.mark.parametrize("name", sorted(BUILDERS))
def test_same_seed_same_bytes(name):
    a, b = _arrays(BUILDERS[name](21)), _arrays(BUILDERS[name](21))
    assert a.keys() == b.keys() and a
    for k in a:
        assert a[k].dtype == b[k].dtype and np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("name", sorted(BUILDERS))
def test_other_seed_other_bytes(name):
    a, b = _arrays(BUILDERS[name](21)), _arrays(BUILDERS[name](22))
    assert any(a[k].shape != b[k].shape or not np.array_equal(a[k], b[k]) for k in a)


def test_freqs_table_is_the_plain_rotary_table():
    """freqs_cis row p: interleaved (cos, sin) of p * base^(-2k/D), computed in
    float64 and rounded once to fp32."""
    t = W.rope_table(16, 8, 10000.0)
    theta = 10000.0 ** (-2.0 * np.arange(4) / 8)
    ang = np.arange(16)[:, None] * theta[None, :]
    assert np.array_equal(t[:, 0::2], np.cos(ang).astype(np.float32))
    assert np.array_equal(t[:, 1::2], np.sin(ang).astype(np.float32))
