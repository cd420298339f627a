"""Seeded sweep over random small configurations of every cache-writing entry
point, each checked against the oracle like the parity tests (values within
the tolerances, untouched bytes bit-exact, guard regions intact, equal error
flags).  The shapes stay inside the documented limits; the point is the
combinations no hand-written case covers (odd head counts with FP8 scales,
padded layouts with mrope sections, subsets that are not whole vectors...).
"""
import numpy as np
import pytest

from gqa_kv_cache_mla_gb300 import workloads as W
from test_gpu_parity import dev, run_gqa, run_knorm, run_mla  # noqa: F401 (dev: fixture)

pytestmark = pytest.mark.gpu

CASES = 12


def _lengths(rng, lo_new=0, hi_new=40, hi_prior=200):
    B = int(rng.integers(1, 13))
    new = rng.integers(lo_new, hi_new + 1, B)
    new[rng.random(B) < 0.2] = 0  # some requests without new tokens
    prior = rng.integers(0, hi_prior + 1, B)
    return new, prior


@pytest.mark.parametrize("case", range(CASES))
def test_mla_random_configurations(orc, dev, case):
    import dataclasses

    rng = np.random.default_rng(7000 + case)
    new, prior = _lengths(rng)
    dtype = W.DTYPE_FP8_E4M3 if rng.random() < 0.5 else W.DTYPE_BF16
    layers = int(rng.integers(1, 4))
    page = int(rng.choice([8, 16, 32, 64]))
    max_seq = int(-(-int((new + prior).max() + 1) // page) * page)
    w = W.mla_workload("sweep", 7100 + case, new, prior, num_heads=int(rng.choice([1, 2, 3, 5, 8])),
                       page_size=page, max_seq_len=max_seq, cache_dtype=dtype,
                       num_layers=layers, layer_idx=int(rng.integers(0, layers)),
                       scale=float(rng.choice([1.0, 0.5, 2.0])) if dtype else 1.0,
                       spare_pages=int(rng.integers(0, 3)))
    if rng.random() < 0.4:
        w = dataclasses.replace(w, q_out_dtype=W.DTYPE_FP8_E4M3)
    if rng.random() < 0.4:
        w = W.mla_inplace(w)
    run_mla(orc, dev, w)


@pytest.mark.parametrize("case", range(CASES))
def test_gqa_random_configurations(orc, dev, case):
    rng = np.random.default_rng(8000 + case)
    new, prior = _lengths(rng, hi_new=30, hi_prior=100)
    S = int(rng.choice([16, 32, 64, 128]))
    Hk = int(rng.choice([1, 2, 4]))
    Hq = Hk * int(rng.choice([1, 2, 4]))
    mode = rng.choice(["slot", "ids", "mrope"])
    sec = None
    if mode == "mrope":
        cuts = np.sort(rng.integers(0, S // 2 + 1, 2))
        sec = (int(cuts[0]), int(cuts[1] - cuts[0]), int(S // 2 - cuts[1]))
    fp8 = rng.random() < 0.4
    w = W.gqa_workload("sweep", 8100 + case, new, prior, Hq, Hk, S,
                       page_size=int(rng.choice([8, 16, 32])), freqs_rows=256, base=10000.0,
                       interleaved=bool(rng.random() < 0.5),
                       position_mode=None if mode == "slot" else str(mode), mrope_section=sec,
                       cache_dtype=W.DTYPE_FP8_E4M3 if fp8 else W.DTYPE_BF16,
                       scale=float(rng.choice([1.0, 0.5])) if fp8 else 1.0,
                       spare_pages=int(rng.integers(0, 3)))
    if rng.random() < 0.3:  # padded layout: 16 spare bytes-multiples after each head / token row
        pad = 16 if fp8 else 8
        w.cache = W.repad_cache(w.cache, pad, 2 * pad, rng)
    run_gqa(orc, dev, w)


@pytest.mark.parametrize("case", range(CASES))
def test_knorm_random_configurations(orc, dev, case):
    rng = np.random.default_rng(9000 + case)
    new, prior = _lengths(rng, hi_new=30, hi_prior=100)
    S = int(rng.choice([8, 16, 64, 128, 256]))
    Hk = int(rng.integers(1, 9))
    per_head = bool(rng.random() < 0.7 or Hk * S > 2048)
    G = int(rng.integers(1, S + 1)) if per_head else Hk * S
    w = W.knorm_workload("sweep", 9100 + case, new, prior, Hk, S,
                         page_size=int(rng.choice([8, 16, 64])), gamma_len=G,
                         weight_offset=float(rng.choice([0.0, 0.5])),
                         multiply_before_cast=bool(rng.random() < 0.6),
                         spare_pages=int(rng.integers(0, 3)), per_head_norm=per_head)
    run_knorm(orc, dev, w, per_head_norm=per_head)
