/*
 * CPU oracle for the fused per-token KV-cache write path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * statement of what the library's entry points compute.  Only the test suite,
 * the package smoke check and the benchmark's CPU-baseline leg load it; the
 * CUDA library never calls, links or includes it, and it shares no code,
 * header, table or helper with the CUDA sources.
 *
 * Precision: every value is widened exactly to fp32 and all arithmetic is
 * IEEE fp32, one operation at a time, in the order the definitions below
 * give (compile with -ffp-contract=off so no multiply-add is fused).
 * Results are rounded once, to the output type.
 *
 * Sources (Modular MAX kernel API pages):
 *  - "mla_fused_rope_rmsnorm_quantization" (Mojo function): description of
 *    the three fused operations; Args q_rope_output, q_rope,
 *    input_row_offsets, freqs_cis, gamma, kv_collection, layer_idx, epsilon;
 *    Parameters kv_input_fn.
 *  - "mla_graph" (Mojo module): module description (dynamic FP8 scaling);
 *    Functions list, entries fused_rope_rmsnorm_quantization_kernel (quantise
 *    before the cache write), fused_rope_rmsnorm_kernel (the in-place
 *    variant), mla_prefill_branch_fp8 (copy the latent values out of the
 *    paged cache, then quantise them) and convert_bf16_to_fp8_e4m3fn.
 *  - "generic_fused_qk_rope_bshd_paged_ragged" (Mojo function): description
 *    (Q rotated into output, K rotated in the paged cache); Parameters
 *    interleaved, has_position_ids, mrope_section; Args q_proj,
 *    input_row_offsets, kv_collection, freqs_cis, position_ids, layer_idx,
 *    output.
 *  - "rms_norm_kv_cache_ragged_paged" (Mojo function): description (in-place
 *    RMSNorm of new K entries located through input_row_offsets, subset of
 *    leading columns given by the length of gamma, weight_offset added to
 *    gamma, multiply_before_cast), parameter per_head_norm.
 *
 * Format sources: bf16 = the upper half of IEEE-754 binary32 with
 * round-to-nearest-even; E4M3FN = OCP 8-bit floating point specification
 * (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * NaN = S.1111.111, largest finite 448, subnormal quantum 2^-9).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - freqs_cis row p holds interleaved (cos, sin) pairs: entry [p][2k] is
 *    the cosine and [p][2k+1] the sine for rotary pair k.
 *  - interleaved=true pairs elements (2k, 2k+1); false pairs (k, k + S/2).
 *    MLA rope parts always use adjacent pairs.
 *  - new token i of request b sits at cache slot pos = cache_lengths[b] + i.
 *  - mrope sections count rotary pairs and sum to S/2; pair k takes its
 *    position from row sec(k) of position_ids[3][T].
 *  - FP8 cache values are stored as satfinite_rne(y / scale).
 *  - multiply_before_cast=false rounds the normalised value to the cache
 *    type first and then multiplies by the weight (a reading the pages do
 *    not fix; pinned by its power-of-two-weight special case).
 *  - per_head_norm=false normalises the whole K row of a token
 *    (num_heads * head_size values) with a gamma of that length (a reading
 *    the pages do not fix; pinned against a float64 library norm).
 *
 * Error flags (returned, OR of):
 *   1 = a slot maps to no valid page (page index past the table, or a page
 *       id >= num_pages including the 0xFFFFFFFF sentinel): that cache row is
 *       not written;
 *   2 = a RoPE position >= freqs rows: nothing of that token is written;
 *   4 = input_row_offsets invalid (first != 0, last != T or decreasing):
 *       nothing at all is written.
 * With T == 0 nothing is examined and 0 is returned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_FLAG_PAGE 1u
#define ORC_FLAG_POS 2u
#define ORC_FLAG_OFFSETS 4u

#define ORC_BF16 0
#define ORC_FP8_E4M3 1

/* ------------------------------------------------------------------ codecs */

float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round an fp32 value to the nearest bf16, ties to the even pattern. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN stays NaN (quiet) */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u; /* may carry into the exponent: correct, up to +inf */
    return (uint16_t)keep;
}

/* Value of an E4M3FN code. */
float oracle_e4m3_to_f32(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int m = c & 7;
    double v;
    if (e == 0xf && m == 7)
        return sign ? -NAN : NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* subnormal: m * 2^-9 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return (float)(sign ? -v : v);
}

/* fp32 -> E4M3FN, round to nearest even, saturating to +-448.  NaN -> NaN. */
uint8_t oracle_f32_to_e4m3(float f) {
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    if (isnan(f))
        return sign | 0x7f;
    double a = fabs((double)f);
    if (a >= 448.0)
        return sign | 0x7e; /* satfinite (also for +-inf) */
    /* quantum of the binade holding a; subnormal binade below 2^-6 */
    double q;
    if (a < ldexp(1.0, -6)) {
        q = ldexp(1.0, -9);
    } else {
        int ex;
        frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) -> floor(log2 a) = ex-1 */
        q = ldexp(1.0, (ex - 1) - 3);
    }
    double n = a / q;         /* exact: division by a power of two */
    double r = nearbyint(n);  /* default mode: ties to even */
    double v = r * q;
    if (v > 448.0)
        v = 448.0; /* cannot happen below 448, kept for clarity */
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6)) /* subnormal: mantissa counts quanta of 2^-9 */
        return sign | (uint8_t)(int)(v / ldexp(1.0, -9));
    int ex;
    double fr = frexp(v, &ex); /* v = fr * 2^ex */
    int e = (ex - 1) + 7;
    int m = (int)((fr * 2.0 - 1.0) * 8.0);
    return sign | (uint8_t)(e << 3) | (uint8_t)m;
}

void oracle_bf16_encode(const float* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(x[i]);
}
void oracle_bf16_decode(const uint16_t* x, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(x[i]);
}
void oracle_e4m3_encode(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_e4m3(x[i]);
}
void oracle_e4m3_decode(const uint8_t* x, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f32(x[i]);
}

/* ------------------------------------------------------------ math steps */

/* Rotate one pair by the angle whose cosine is c and sine is s:
 * (y0, y1) = (x0*c - x1*s, x0*s + x1*c); each product rounded to fp32, then
 * the sum rounded to fp32. */
static void rope_pair(float x0, float x1, float c, float s, float* y0, float* y1) {
    float x0c = x0 * c;
    float x1s = x1 * s;
    float x0s = x0 * s;
    float x1c = x1 * c;
    *y0 = x0c - x1s;
    *y1 = x0s + x1c;
}

/* Exported for the tests: rotate n pairs x[2k], x[2k+1] by cs[2k] (cos),
 * cs[2k+1] (sin), fp32 in and out. */
void oracle_rope_pairs_f32(const float* x, const float* cs, float* y, int64_t n_pairs) {
    for (int64_t k = 0; k < n_pairs; ++k)
        rope_pair(x[2 * k], x[2 * k + 1], cs[2 * k], cs[2 * k + 1], &y[2 * k], &y[2 * k + 1]);
}

/* 1 / sqrt(mean(x^2) + eps): squares summed left to right in fp32. */
float oracle_rms_inv(const float* x, int64_t n, float eps) {
    float ss = 0.0f;
    for (int64_t j = 0; j < n; ++j) {
        float sq = x[j] * x[j];
        ss = ss + sq;
    }
    float mean = ss / (float)n;
    float d = sqrtf(mean + eps);
    return 1.0f / d;
}

/* Exported for the tests: y = (x * r) * w in fp32, r = oracle_rms_inv. */
void oracle_rms_norm_f32(const float* x, const float* w, int64_t n, float eps, float* y) {
    float r = oracle_rms_inv(x, n, eps);
    for (int64_t j = 0; j < n; ++j) {
        float xr = x[j] * r;
        y[j] = xr * w[j];
    }
}

/* one fp32 value into a cache element of the given type */
static void store_elem(void* base, int64_t idx, int dtype, float scale, float y) {
    if (dtype == ORC_BF16) {
        ((uint16_t*)base)[idx] = oracle_f32_to_bf16(y);
    } else {
        float z = y / scale;
        ((uint8_t*)base)[idx] = oracle_f32_to_e4m3(z);
    }
}

/* ---------------------------------------------------------- ragged lookup */

/* Offsets must start at 0, never decrease and end at T. */
static int offsets_valid(const uint32_t* offsets, uint32_t B, uint32_t T) {
    if (offsets[0] != 0u || offsets[B] != T) return 0;
    for (uint32_t b = 0; b < B; ++b)
        if (offsets[b] > offsets[b + 1]) return 0;
    return 1;
}

/* For each token t: its request b and index i inside the request, by walking
 * the requests in order (request b owns tokens offsets[b] .. offsets[b+1]-1). */
static void token_map(const uint32_t* offsets, uint32_t B, uint32_t* tok_b, uint32_t* tok_i) {
    for (uint32_t b = 0; b < B; ++b)
        for (uint32_t t = offsets[b]; t < offsets[b + 1]; ++t) {
            tok_b[t] = b;
            tok_i[t] = t - offsets[b];
        }
}

/* Cache element index of (page, kv=0 (K), layer, row, head, col=0), or -1 with
 * *flags |= PAGE when the slot maps to no valid page. */
typedef struct {
    uint32_t num_pages, num_layers, page_size, num_heads, head_size, max_pages;
    int64_t s_page, s_kv, s_layer, s_token, s_head;
    const uint32_t* page_table;
} orc_layout;

static int64_t slot_base(const orc_layout* L, uint32_t b, uint64_t pos, uint32_t layer,
                         uint32_t* flags) {
    uint64_t pidx = pos / L->page_size;
    if (pidx >= L->max_pages) {
        *flags |= ORC_FLAG_PAGE;
        return -1;
    }
    uint32_t page = L->page_table[(uint64_t)b * L->max_pages + pidx];
    if (page >= L->num_pages) {
        *flags |= ORC_FLAG_PAGE;
        return -1;
    }
    uint64_t row = pos % L->page_size;
    return (int64_t)page * L->s_page + (int64_t)layer * L->s_layer + (int64_t)row * L->s_token;
}

/* -------------------------------------------------------------- MLA path */

/*
 * mla_fused_rope_rmsnorm_quantization, for every new token t of request b at
 * slot position pos = cache_lengths[b] + i:
 *   1. RoPE on q_rope[t, h, :] (64 values = 32 adjacent pairs) with
 *      freqs_cis[pos] -> q_rope_output[t, h, :] (bf16), every head h;
 *      RoPE on the rope part kv_in[t, 512:576] with the same row;
 *   2. RMSNorm of the non-rope part kv_in[t, 0:512] with gamma and epsilon;
 *   3. the 576-wide result quantised to the cache type and written to the
 *      cache row of slot pos in layer layer_idx (head 0).
 */
uint32_t oracle_mla_rope_rmsnorm_quant(
    void* q_rope_out, int out_dtype, const uint16_t* q_rope, const uint32_t* offsets, uint32_t B,
    uint32_t T, uint32_t H, const float* freqs, uint32_t freqs_rows, const uint16_t* gamma,
    const uint16_t* kv_in, int64_t kv_row_stride, void* cache, int cache_dtype, float scale,
    const uint32_t* page_table, uint32_t max_pages, const uint32_t* cache_lengths,
    uint32_t num_pages, uint32_t num_layers, uint32_t page_size, uint32_t num_heads,
    uint32_t head_size, int64_t s_page, int64_t s_kv, int64_t s_layer, int64_t s_token,
    int64_t s_head, uint32_t layer_idx, float eps, int nthreads) {
    const uint32_t NORM = 512, ROPE = 64, ROW = 576;
    (void)num_layers;
    (void)num_heads;
    (void)head_size;
    (void)s_kv;
    (void)s_head;
    if (T == 0) return 0;
    if (!offsets_valid(offsets, B, T)) return ORC_FLAG_OFFSETS;
    orc_layout L = {num_pages, num_layers, page_size, num_heads, head_size, max_pages,
                    s_page, s_kv, s_layer, s_token, s_head, page_table};
    uint32_t* tok_b = (uint32_t*)malloc(sizeof(uint32_t) * T);
    uint32_t* tok_i = (uint32_t*)malloc(sizeof(uint32_t) * T);
    token_map(offsets, B, tok_b, tok_i);
    float g[512];
    for (uint32_t j = 0; j < NORM; ++j) g[j] = oracle_bf16_to_f32(gamma[j]);
    uint32_t flags = 0;
    int64_t t;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) reduction(| : flags) schedule(static)
    for (t = 0; t < (int64_t)T; ++t) {
        uint32_t b = tok_b[t];
        uint64_t pos = (uint64_t)cache_lengths[b] + tok_i[t];
        if (pos >= freqs_rows) {
            flags |= ORC_FLAG_POS;
            continue;
        }
        const float* cs = freqs + pos * ROPE;
        /* 1a. q rope, every head */
        for (uint32_t h = 0; h < H; ++h) {
            const uint16_t* xq = q_rope + ((int64_t)t * H + h) * ROPE;
            const int64_t yo = ((int64_t)t * H + h) * ROPE;
            for (uint32_t k = 0; k < ROPE / 2; ++k) {
                float y0, y1;
                rope_pair(oracle_bf16_to_f32(xq[2 * k]), oracle_bf16_to_f32(xq[2 * k + 1]),
                          cs[2 * k], cs[2 * k + 1], &y0, &y1);
                /* bf16, or E4M3 by direct saturating conversion (no scale) */
                store_elem(q_rope_out, yo + 2 * k, out_dtype, 1.0f, y0);
                store_elem(q_rope_out, yo + 2 * k + 1, out_dtype, 1.0f, y1);
            }
        }
        /* the cache row this token writes */
        uint32_t f = 0;
        int64_t base = slot_base(&L, b, pos, layer_idx, &f);
        flags |= f;
        if (base < 0) continue;
        const uint16_t* xr = kv_in + (int64_t)t * kv_row_stride;
        float row[576];
        for (uint32_t j = 0; j < ROW; ++j) row[j] = oracle_bf16_to_f32(xr[j]);
        float y[576];
        /* 1b. k rope part */
        for (uint32_t k = 0; k < ROPE / 2; ++k)
            rope_pair(row[NORM + 2 * k], row[NORM + 2 * k + 1], cs[2 * k], cs[2 * k + 1],
                      &y[NORM + 2 * k], &y[NORM + 2 * k + 1]);
        /* 2. RMSNorm of the latent part */
        oracle_rms_norm_f32(row, g, NORM, eps, y);
        /* 3. quantise and write */
        for (uint32_t j = 0; j < ROW; ++j) store_elem(cache, base + j, cache_dtype, scale, y[j]);
    }
    free(tok_b);
    free(tok_i);
    return flags;
}

/* Value of cache element idx: bf16 widened, or E4M3 decoded times scale. */
static float load_elem(const void* base, int64_t idx, int dtype, float scale) {
    if (dtype == ORC_BF16) return oracle_bf16_to_f32(((const uint16_t*)base)[idx]);
    return oracle_e4m3_to_f32(((const uint8_t*)base)[idx]) * scale;
}

/*
 * fused_rope_rmsnorm_kernel ("mla_graph" module page; first two steps of the
 * MLA decode and prefill branches): the same computation as above, but the
 * 576-wide latent rows of the new tokens are already in the cache (written by
 * the latent projection) and are normalised and rotated in place; the cache
 * may be bf16 or FP8 E4M3 (dequantised with its scale, re-quantised after).
 */
uint32_t oracle_mla_rope_rmsnorm_inplace(
    void* q_rope_out, int out_dtype, const uint16_t* q_rope, const uint32_t* offsets, uint32_t B,
    uint32_t T, uint32_t H, const float* freqs, uint32_t freqs_rows, const uint16_t* gamma,
    void* cache, int cache_dtype, float scale, const uint32_t* page_table, uint32_t max_pages,
    const uint32_t* cache_lengths, uint32_t num_pages, uint32_t num_layers, uint32_t page_size,
    int64_t s_page, int64_t s_layer, int64_t s_token, uint32_t layer_idx, float eps, int nthreads) {
    const uint32_t NORM = 512, ROPE = 64, ROW = 576;
    if (T == 0) return 0;
    if (!offsets_valid(offsets, B, T)) return ORC_FLAG_OFFSETS;
    orc_layout L = {num_pages, num_layers, page_size, 1, ROW, max_pages,
                    s_page, 0, s_layer, s_token, ROW, page_table};
    uint32_t* tok_b = (uint32_t*)malloc(sizeof(uint32_t) * T);
    uint32_t* tok_i = (uint32_t*)malloc(sizeof(uint32_t) * T);
    token_map(offsets, B, tok_b, tok_i);
    float g[512];
    for (uint32_t j = 0; j < NORM; ++j) g[j] = oracle_bf16_to_f32(gamma[j]);
    uint32_t flags = 0;
    int64_t t;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) reduction(| : flags) schedule(static)
    for (t = 0; t < (int64_t)T; ++t) {
        uint32_t b = tok_b[t];
        uint64_t pos = (uint64_t)cache_lengths[b] + tok_i[t];
        if (pos >= freqs_rows) {
            flags |= ORC_FLAG_POS;
            continue;
        }
        const float* cs = freqs + pos * ROPE;
        for (uint32_t h = 0; h < H; ++h) {
            const uint16_t* xq = q_rope + ((int64_t)t * H + h) * ROPE;
            const int64_t yo = ((int64_t)t * H + h) * ROPE;
            for (uint32_t k = 0; k < ROPE / 2; ++k) {
                float y0, y1;
                rope_pair(oracle_bf16_to_f32(xq[2 * k]), oracle_bf16_to_f32(xq[2 * k + 1]),
                          cs[2 * k], cs[2 * k + 1], &y0, &y1);
                store_elem(q_rope_out, yo + 2 * k, out_dtype, 1.0f, y0);
                store_elem(q_rope_out, yo + 2 * k + 1, out_dtype, 1.0f, y1);
            }
        }
        uint32_t f = 0;
        int64_t base = slot_base(&L, b, pos, layer_idx, &f);
        flags |= f;
        if (base < 0) continue;
        float row[576], y[576];
        for (uint32_t j = 0; j < ROW; ++j) row[j] = load_elem(cache, base + j, cache_dtype, scale);
        for (uint32_t k = 0; k < ROPE / 2; ++k)
            rope_pair(row[NORM + 2 * k], row[NORM + 2 * k + 1], cs[2 * k], cs[2 * k + 1],
                      &y[NORM + 2 * k], &y[NORM + 2 * k + 1]);
        oracle_rms_norm_f32(row, g, NORM, eps, y);
        for (uint32_t j = 0; j < ROW; ++j) store_elem(cache, base + j, cache_dtype, scale, y[j]);
    }
    free(tok_b);
    free(tok_i);
    return flags;
}

/*
 * convert_bf16_to_fp8_e4m3fn ("mla_graph" module page): n bf16 values to
 * E4M3 codes, satfinite_rne(x / scale).
 */
void oracle_convert_bf16_to_e4m3(const uint16_t* in, uint8_t* out, int64_t n, float scale) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_e4m3(oracle_bf16_to_f32(in[i]) / scale);
}

/*
 * Dynamic FP8 scaling ("mla_graph" module page), per row (token): the scale
 * of a row is amax(|x|) / 448 (1 for an all-zero row) and its codes are
 * satfinite_rne(x / scale), so the row's largest magnitude maps to 448.
 */
void oracle_quantize_rows_e4m3(const uint16_t* in, int64_t in_stride, uint8_t* out,
                               int64_t out_stride, float* scales, int64_t rows, int64_t cols) {
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(oracle_bf16_to_f32(in[r * in_stride + c]));
            if (a > amax) amax = a;
        }
        float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        scales[r] = sc;
        for (int64_t c = 0; c < cols; ++c)
            out[r * out_stride + c] = oracle_f32_to_e4m3(oracle_bf16_to_f32(in[r * in_stride + c]) / sc);
    }
}

/*
 * Paged -> contiguous copy of the MLA latent cache (the step after the
 * in-place RoPE/RMSNorm in the FP8 prefill branch): request b's context rows
 * (positions 0 .. ctx_offsets[b+1] - ctx_offsets[b] - 1 of its cache) are
 * copied to out rows ctx_offsets[b] .. ctx_offsets[b+1]-1, converted from
 * the cache type (bf16, or E4M3 times cache_scale) to the output type (bf16
 * round to nearest even, or E4M3 satfinite_rne(v / out_scale)).  Flags:
 * 4 when ctx_offsets do not start at 0, decrease or do not end at rows;
 * 1 for a row without a valid page (the row is not written).
 */
uint32_t oracle_mla_gather_latent(void* out, int out_dtype, float out_scale, const void* cache,
                                  int cache_dtype, float cache_scale, const uint32_t* page_table,
                                  uint32_t max_pages, uint32_t num_pages, uint32_t num_layers,
                                  uint32_t page_size, int64_t s_page, int64_t s_layer,
                                  int64_t s_token, uint32_t layer_idx, const uint32_t* ctx_offsets,
                                  uint32_t B, uint32_t rows) {
    const uint32_t ROW = 576;
    if (rows == 0) return 0;
    if (!offsets_valid(ctx_offsets, B, rows)) return ORC_FLAG_OFFSETS;
    orc_layout L = {num_pages, num_layers, page_size, 1, ROW, max_pages,
                    s_page, 0, s_layer, s_token, ROW, page_table};
    uint32_t flags = 0;
    for (uint32_t b = 0; b < B; ++b) {
        for (uint32_t r = ctx_offsets[b]; r < ctx_offsets[b + 1]; ++r) {
            uint64_t pos = r - ctx_offsets[b];
            uint32_t f = 0;
            int64_t base = slot_base(&L, b, pos, layer_idx, &f);
            flags |= f;
            if (base < 0) continue;
            for (uint32_t j = 0; j < ROW; ++j)
                store_elem(out, (int64_t)r * ROW + j, out_dtype, out_scale,
                           load_elem(cache, base + j, cache_dtype, cache_scale));
        }
    }
    return flags;
}

/*
 * The same copy with dynamic per-row FP8 (the quantisation of the FP8
 * prefill branch with dynamic scaling, one scale per context row): the 576
 * values of the row as the cache holds them (bf16, or E4M3 times
 * cache_scale), scale = max|v| / 448 (1 for a row of zeros), codes =
 * satfinite_rne(v / scale).  Rows without a valid page are not written
 * (neither their codes nor their scale).  Flags as the plain copy.
 */
uint32_t oracle_mla_gather_latent_dynamic(uint8_t* out, float* scales, const void* cache,
                                          int cache_dtype, float cache_scale,
                                          const uint32_t* page_table, uint32_t max_pages,
                                          uint32_t num_pages, uint32_t num_layers,
                                          uint32_t page_size, int64_t s_page, int64_t s_layer,
                                          int64_t s_token, uint32_t layer_idx,
                                          const uint32_t* ctx_offsets, uint32_t B,
                                          uint32_t rows) {
    const uint32_t ROW = 576;
    if (rows == 0) return 0;
    if (!offsets_valid(ctx_offsets, B, rows)) return ORC_FLAG_OFFSETS;
    orc_layout L = {num_pages, num_layers, page_size, 1, ROW, max_pages,
                    s_page, 0, s_layer, s_token, ROW, page_table};
    uint32_t flags = 0;
    float v[576];
    for (uint32_t b = 0; b < B; ++b) {
        for (uint32_t r = ctx_offsets[b]; r < ctx_offsets[b + 1]; ++r) {
            uint64_t pos = r - ctx_offsets[b];
            uint32_t f = 0;
            int64_t base = slot_base(&L, b, pos, layer_idx, &f);
            flags |= f;
            if (base < 0) continue;
            float amax = 0.0f;
            for (uint32_t j = 0; j < ROW; ++j) {
                v[j] = load_elem(cache, base + j, cache_dtype, cache_scale);
                float a = fabsf(v[j]);
                if (a > amax) amax = a;
            }
            float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[r] = sc;
            for (uint32_t j = 0; j < ROW; ++j)
                out[(int64_t)r * ROW + j] = oracle_f32_to_e4m3(v[j] / sc);
        }
    }
    return flags;
}

/* -------------------------------------------------------------- GQA path */

/* Position used for rotary pair k of token t (cache slot position pos_s when
 * no position_ids are given). */
static uint64_t pair_position(uint64_t pos_s, const uint32_t* position_ids, const uint32_t* sec,
                              uint32_t T, int64_t t, uint32_t k) {
    if (!position_ids) return pos_s;
    if (!sec) return position_ids[t];
    uint32_t row = (k < sec[0]) ? 0u : (k < sec[0] + sec[1]) ? 1u : 2u;
    return position_ids[(int64_t)row * T + t];
}

/* Element indices of pair k inside a head of size S. */
static void pair_elems(int interleaved, uint32_t S, uint32_t k, uint32_t* e0, uint32_t* e1) {
    if (interleaved) {
        *e0 = 2 * k;
        *e1 = 2 * k + 1;
    } else {
        *e0 = k;
        *e1 = k + S / 2;
    }
}

static void rotate_head_bf16(const uint16_t* x, uint16_t* y, uint32_t S, int interleaved,
                             const float* freqs, uint64_t pos_s, const uint32_t* position_ids,
                             const uint32_t* sec, uint32_t T, int64_t t) {
    uint16_t out[1024];
    for (uint32_t k = 0; k < S / 2; ++k) {
        uint32_t e0, e1;
        pair_elems(interleaved, S, k, &e0, &e1);
        uint64_t p = pair_position(pos_s, position_ids, sec, T, t, k);
        const float* cs = freqs + p * S;
        float y0, y1;
        rope_pair(oracle_bf16_to_f32(x[e0]), oracle_bf16_to_f32(x[e1]), cs[2 * k], cs[2 * k + 1],
                  &y0, &y1);
        out[e0] = oracle_f32_to_bf16(y0);
        out[e1] = oracle_f32_to_bf16(y1);
    }
    memcpy(y, out, sizeof(uint16_t) * S); /* safe when y == x */
}

/* The same rotation on an FP8 E4M3 head row stored with a per-tensor scale:
 * each value is dequantised (code value times scale, rounded to fp32),
 * rotated, and re-encoded as satfinite_rne(y / scale). */
static void rotate_head_e4m3(uint8_t* x, uint32_t S, int interleaved, float scale,
                             const float* freqs, uint64_t pos_s, const uint32_t* position_ids,
                             const uint32_t* sec, uint32_t T, int64_t t) {
    uint8_t out[1024];
    for (uint32_t k = 0; k < S / 2; ++k) {
        uint32_t e0, e1;
        pair_elems(interleaved, S, k, &e0, &e1);
        uint64_t p = pair_position(pos_s, position_ids, sec, T, t, k);
        const float* cs = freqs + p * S;
        float x0 = oracle_e4m3_to_f32(x[e0]) * scale;
        float x1 = oracle_e4m3_to_f32(x[e1]) * scale;
        float y0, y1;
        rope_pair(x0, x1, cs[2 * k], cs[2 * k + 1], &y0, &y1);
        out[e0] = oracle_f32_to_e4m3(y0 / scale);
        out[e1] = oracle_f32_to_e4m3(y1 / scale);
    }
    memcpy(x, out, S);
}

/*
 * generic_fused_qk_rope_bshd_paged_ragged: for every new token t, Q heads
 * q_proj[t, h, :] are rotated into output[t, h, :]; the K rows of the token's
 * slot (all kv heads, layer layer_idx) are rotated in place in the cache
 * (bf16, or FP8 E4M3 with a per-tensor scale: the collection's scale_dtype_ /
 * quantization_granularity_ parameters).
 */
uint32_t oracle_qk_rope_paged_ragged(
    const uint16_t* q_proj, const uint32_t* offsets, uint32_t B, uint32_t T, uint32_t Hq,
    void* cache, int cache_dtype, float scale, const uint32_t* page_table, uint32_t max_pages,
    const uint32_t* cache_lengths, uint32_t num_pages, uint32_t num_layers, uint32_t page_size,
    uint32_t num_kv_heads, uint32_t head_size, int64_t s_page, int64_t s_kv, int64_t s_layer,
    int64_t s_token, int64_t s_head, const float* freqs, uint32_t freqs_rows,
    const uint32_t* position_ids, int interleaved, const uint32_t* mrope_section,
    uint32_t layer_idx, uint16_t* output, int nthreads) {
    const uint32_t S = head_size;
    if (T == 0) return 0;
    if (!offsets_valid(offsets, B, T)) return ORC_FLAG_OFFSETS;
    orc_layout L = {num_pages, num_layers, page_size, num_kv_heads, head_size, max_pages,
                    s_page, s_kv, s_layer, s_token, s_head, page_table};
    uint32_t* tok_b = (uint32_t*)malloc(sizeof(uint32_t) * T);
    uint32_t* tok_i = (uint32_t*)malloc(sizeof(uint32_t) * T);
    token_map(offsets, B, tok_b, tok_i);
    uint32_t flags = 0;
    int64_t t;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) reduction(| : flags) schedule(static)
    for (t = 0; t < (int64_t)T; ++t) {
        uint32_t b = tok_b[t];
        uint64_t pos_s = (uint64_t)cache_lengths[b] + tok_i[t];
        int bad = 0;
        for (uint32_t k = 0; k < S / 2; ++k)
            if (pair_position(pos_s, position_ids, mrope_section, T, t, k) >= freqs_rows) bad = 1;
        if (bad) {
            flags |= ORC_FLAG_POS;
            continue;
        }
        for (uint32_t h = 0; h < Hq; ++h)
            rotate_head_bf16(q_proj + ((int64_t)t * Hq + h) * S, output + ((int64_t)t * Hq + h) * S,
                             S, interleaved, freqs, pos_s, position_ids, mrope_section, T, t);
        uint32_t f = 0;
        int64_t base = slot_base(&L, b, pos_s, layer_idx, &f);
        flags |= f;
        if (base < 0) continue;
        for (uint32_t g = 0; g < num_kv_heads; ++g) { /* kv index 0 = K */
            if (cache_dtype == ORC_BF16) {
                uint16_t* k = (uint16_t*)cache + base + (int64_t)g * s_head;
                rotate_head_bf16(k, k, S, interleaved, freqs, pos_s, position_ids, mrope_section, T,
                                 t);
            } else {
                uint8_t* k = (uint8_t*)cache + base + (int64_t)g * s_head;
                rotate_head_e4m3(k, S, interleaved, scale, freqs, pos_s, position_ids,
                                 mrope_section, T, t);
            }
        }
    }
    free(tok_b);
    free(tok_i);
    return flags;
}

/* ------------------------------------------------------ K-cache RMSNorm */

/* RMSNorm of n values read from src (bf16) written back to dst, weight
 * w_j = gamma_j + weight_offset. */
static void rms_norm_bf16(const uint16_t* const* src, uint16_t* const* dst, int64_t n,
                          const float* w, float eps, int multiply_before_cast) {
    float xs[8192];
    for (int64_t j = 0; j < n; ++j) xs[j] = oracle_bf16_to_f32(*src[j]);
    float r = oracle_rms_inv(xs, n, eps);
    for (int64_t j = 0; j < n; ++j) {
        float xr = xs[j] * r;
        float y;
        if (multiply_before_cast) {
            y = xr * w[j];
        } else {
            float xr_c = oracle_bf16_to_f32(oracle_f32_to_bf16(xr));
            y = xr_c * w[j];
        }
        *dst[j] = oracle_f32_to_bf16(y);
    }
}

/*
 * rms_norm_kv_cache_ragged_paged: for every new token t (slot pos_s) and, with
 * per_head_norm, every kv head g: the leading gamma_len columns of the K row
 * are RMS-normalised in place; columns >= gamma_len are left as they are.
 * Without per_head_norm the whole num_heads*head_size K row is normalised as
 * one vector and gamma_len must equal that width.
 */
uint32_t oracle_rms_norm_kv_cache_paged(
    uint16_t* cache, const uint32_t* page_table, uint32_t max_pages,
    const uint32_t* cache_lengths, uint32_t num_pages, uint32_t num_layers, uint32_t page_size,
    uint32_t num_kv_heads, uint32_t head_size, int64_t s_page, int64_t s_kv, int64_t s_layer,
    int64_t s_token, int64_t s_head, const uint16_t* gamma, uint32_t gamma_len, float eps,
    float weight_offset, uint32_t layer_idx, uint32_t total_seq_len, const uint32_t* offsets,
    uint32_t B, int multiply_before_cast, int per_head_norm, int nthreads) {
    uint32_t T = total_seq_len;
    if (T == 0) return 0;
    if (!offsets_valid(offsets, B, T)) return ORC_FLAG_OFFSETS;
    if (gamma_len == 0 || gamma_len > 8192) return 0xffffffffu;
    if (per_head_norm && gamma_len > head_size) return 0xffffffffu;
    if (!per_head_norm && gamma_len != num_kv_heads * head_size) return 0xffffffffu;
    orc_layout L = {num_pages, num_layers, page_size, num_kv_heads, head_size, max_pages,
                    s_page, s_kv, s_layer, s_token, s_head, page_table};
    uint32_t* tok_b = (uint32_t*)malloc(sizeof(uint32_t) * T);
    uint32_t* tok_i = (uint32_t*)malloc(sizeof(uint32_t) * T);
    token_map(offsets, B, tok_b, tok_i);
    float* w = (float*)malloc(sizeof(float) * (gamma_len ? gamma_len : 1));
    for (uint32_t j = 0; j < gamma_len; ++j) w[j] = oracle_bf16_to_f32(gamma[j]) + weight_offset;
    uint32_t flags = 0;
    int64_t t;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) reduction(| : flags) schedule(static)
    for (t = 0; t < (int64_t)T; ++t) {
        uint32_t b = tok_b[t];
        uint64_t pos_s = (uint64_t)cache_lengths[b] + tok_i[t];
        uint32_t f = 0;
        int64_t base = slot_base(&L, b, pos_s, layer_idx, &f);
        flags |= f;
        if (base < 0) continue;
        uint16_t* ptrs_static[8192];
        uint16_t** ptrs = ptrs_static;
        if (per_head_norm) {
            for (uint32_t g = 0; g < num_kv_heads; ++g) {
                for (uint32_t j = 0; j < gamma_len; ++j) ptrs[j] = cache + base + (int64_t)g * s_head + j;
                rms_norm_bf16((const uint16_t* const*)ptrs, ptrs, gamma_len, w, eps,
                              multiply_before_cast);
            }
        } else {
            for (uint32_t g = 0; g < num_kv_heads; ++g)
                for (uint32_t j = 0; j < head_size; ++j)
                    ptrs[(int64_t)g * head_size + j] = cache + base + (int64_t)g * s_head + j;
            rms_norm_bf16((const uint16_t* const*)ptrs, ptrs, (int64_t)num_kv_heads * head_size, w,
                          eps, multiply_before_cast);
        }
    }
    free(w);
    free(tok_b);
    free(tok_i);
    return flags;
}

int oracle_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}
