"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, index, operand or rounding rule), compiles it on the CPU
and runs the pin tests against it: at least one pin must fail.  The real
oracle is never modified.
"""
import os

import pytest

import oracle
import test_oracle_codecs as C
import test_oracle_next as X
import test_oracle_rmsnorm as N
import test_oracle_rope as R
import test_oracle_scatter as S

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("rope sign of the sine term", "*y0 = x0c - x1s;", "*y0 = x0c + x1s;"),
    ("rope cos/sin swapped", "float x0c = x0 * c;", "float x0c = x0 * s;"),
    ("rope second output", "*y1 = x0s + x1c;", "*y1 = x1c - x0s;"),
    ("half-split partner", "*e1 = k + S / 2;", "*e1 = S - 1 - k;"),
    ("mrope section boundary", "(k < sec[0] + sec[1]) ? 1u", "(k <= sec[0] + sec[1]) ? 1u"),
    ("position ids ignored", "if (!sec) return position_ids[t];", "if (!sec) return pos_s;"),
    ("rms eps dropped", "float d = sqrtf(mean + eps);", "float d = sqrtf(mean);"),
    ("rms wrong count", "float mean = ss / (float)n;", "float mean = ss / (float)(n + 1);"),
    ("rms square dropped", "float sq = x[j] * x[j];", "float sq = x[j];"),
    ("gamma index shifted", "y[j] = xr * w[j];", "y[j] = xr * w[(j + 1) % n];"),
    ("weight offset dropped", "+ weight_offset;", "+ 0.0f;"),
    ("slot position off by one",
     "uint64_t pos = (uint64_t)cache_lengths[b] + tok_i[t];",
     "uint64_t pos = (uint64_t)cache_lengths[b] + tok_i[t] + 1;"),
    ("row inside page", "uint64_t row = pos % L->page_size;",
     "uint64_t row = (pos + 1) % L->page_size;"),
    ("layer offset dropped", "(int64_t)layer * L->s_layer", "(int64_t)0 * L->s_layer"),
    ("K rows taken from V", "uint16_t* k = (uint16_t*)cache + base + (int64_t)g * s_head;",
     "uint16_t* k = (uint16_t*)cache + base + s_kv + (int64_t)g * s_head;"),
    ("fp8 K dequantised without the scale", "float x0 = oracle_e4m3_to_f32(x[e0]) * scale;",
     "float x0 = oracle_e4m3_to_f32(x[e0]);"),
    ("fp8 K re-quantised without the scale", "out[e1] = oracle_f32_to_e4m3(y1 / scale);",
     "out[e1] = oracle_f32_to_e4m3(y1);"),
    ("q head order", "const int64_t yo = ((int64_t)t * H + h) * ROPE;",
     "const int64_t yo = ((int64_t)t * H + (H - 1 - h)) * ROPE;"),
    ("bf16 truncates", "keep += 1u;", "keep += 0u;"),
    ("e4m3 ties away from zero", "double r = nearbyint(n);", "double r = round(n);"),
    ("e4m3 subnormal quantum", "q = ldexp(1.0, -9);", "q = ldexp(1.0, -10);"),
    ("fp8 scale multiplies", "float z = y / scale;", "float z = y * scale;"),
    ("q output pair element swapped",
     "store_elem(q_rope_out, yo + 2 * k + 1, out_dtype, 1.0f, y1);",
     "store_elem(q_rope_out, yo + 2 * k + 1, out_dtype, 1.0f, y0);"),
    ("in-place row read without the scale",
     "return oracle_e4m3_to_f32(((const uint8_t*)base)[idx]) * scale;",
     "return oracle_e4m3_to_f32(((const uint8_t*)base)[idx]);"),
    ("convert ignores the scale", "out[i] = oracle_f32_to_e4m3(oracle_bf16_to_f32(in[i]) / scale);",
     "out[i] = oracle_f32_to_e4m3(oracle_bf16_to_f32(in[i]));"),
    ("row scale against the wrong maximum", "float sc = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "float sc = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    ("row maximum of signed values", "float a = fabsf(oracle_bf16_to_f32(in[r * in_stride + c]));",
     "float a = oracle_bf16_to_f32(in[r * in_stride + c]);"),
    ("gather position off by one", "uint64_t pos = r - ctx_offsets[b];",
     "uint64_t pos = r - ctx_offsets[b] + 1;"),
    ("whole-row norm over the first head only",
     "rms_norm_bf16((const uint16_t* const*)ptrs, ptrs, (int64_t)num_kv_heads * head_size, w,",
     "rms_norm_bf16((const uint16_t* const*)ptrs, ptrs, (int64_t)head_size, w,"),
    ("cast-first norm without the intermediate rounding",
     "float xr_c = oracle_bf16_to_f32(oracle_f32_to_bf16(xr));", "float xr_c = xr;"),
    ("dynamic gather ignores the cache scale",
     "v[j] = load_elem(cache, base + j, cache_dtype, cache_scale);",
     "v[j] = load_elem(cache, base + j, cache_dtype, 1.0f);"),
    ("dynamic gather multiplies by its scale",
     "out[(int64_t)r * ROW + j] = oracle_f32_to_e4m3(v[j] / sc);",
     "out[(int64_t)r * ROW + j] = oracle_f32_to_e4m3(v[j] * sc);"),
    ("offsets order unchecked", "if (offsets[b] > offsets[b + 1]) return 0;",
     "if (0) return 0;"),
    ("page id range unchecked", "if (page >= L->num_pages) {", "if (page == 0xffffffffu) {"),
    ("position range unchecked", "if (pos >= freqs_rows) {", "if (pos > freqs_rows) {"),
]

PINS = [
    (C.test_bf16_encode_matches_torch_random, {}),
    (C.test_bf16_encode_ties_and_neighbours, {}),
    (C.test_e4m3_decode_all_codes_match_torch, {}),
    (C.test_e4m3_spec_points, {}),
    (C.test_e4m3_encode_matches_torch_in_range, {}),
    (R.test_rope_pairs_vs_complex_fp64, {}),
    (R.test_mla_q_and_k_rope_vs_complex_fp64, {}),
    (R.test_mla_position_zero_identity, {}),
    (R.test_gqa_half_split_is_permuted_interleaved, {}),
    (N.test_unit_weight_rms_closed_form, {"n": 512, "eps": 0.5}),
    (N.test_rms_norm_vs_torch, {}),
    (N.test_mla_latent_part_vs_torch, {}),
    (N.test_knorm_subset_vs_torch, {"G": 16}),
    (N.test_knorm_weight_offset_adds_to_gamma, {}),
    (N.test_knorm_whole_row_norm, {}),
    (N.test_knorm_multiply_after_cast_within_one_ulp, {}),
    (S.test_mla_tiny_writes_exactly_new_rows, {"dtype": 1}),
    (S.test_gqa_rotates_only_new_k_rows, {}),
    (S.test_knorm_touches_only_leading_cols_of_new_rows, {}),
    (S.test_invalid_offsets_write_nothing, {}),
    (S.test_position_past_table_skips_token, {}),
    (S.test_unmapped_page_skips_cache_row_only, {}),
    (S.test_fp8_scale_convention, {}),
    (R.test_gqa_fp8_k_position_zero_is_identity, {}),
    (X.test_fp8_q_output_vs_complex_fp64, {}),
    (X.test_convert_scale_is_a_division, {"k": 1}),
    (X.test_dynamic_row_quantisation_closed_form, {}),
    (X.test_inplace_equals_fused_write, {"dtype": 1}),
    (X.test_gather_brute_force, {"src": 0, "dst": 1}),
    (X.test_gather_fp8_cache_scale, {}),
    (R.test_gqa_fp8_k_vs_complex_fp64, {"interleaved": False}),
    (R.test_gqa_fp8_k_scale_convention, {}),
    (X.test_gather_dynamic_closed_form_fp8_cache, {}),
] + [(R.test_gqa_q_and_k_vs_complex_fp64, {"interleaved": i, "mode": m})
     for i in (True, False) for m in (None, "ids", "mrope")]


def test_real_oracle_passes_every_listed_pin(orc):
    for fn, kw in PINS:
        fn(orc, **kw)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, name
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new, 1))  # the first occurrence
    v = oracle.Variant(oracle.compile_source(str(path), str(tmp_path / "mutant.so")))
    for fn, kw in PINS:
        try:
            fn(v, **kw)
        except AssertionError:
            return
    pytest.fail("no pin caught the planted mistake: " + name)
