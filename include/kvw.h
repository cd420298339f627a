/*
 * kvw.h - C ABI of the GB300 fused per-token KV-cache write library.
 *
 * One entry point per operation of the Modular MAX kernel pages:
 *   kvw_mla_rope_rmsnorm_quant         "mla_fused_rope_rmsnorm_quantization"
 *   kvw_qk_rope_paged_ragged           "generic_fused_qk_rope_bshd_paged_ragged"
 *   kvw_rms_norm_kv_cache_paged        "rms_norm_kv_cache_ragged_paged"
 * and for the steps of the "mla_graph" module page around them:
 *   kvw_mla_rope_rmsnorm_inplace       fused_rope_rmsnorm_kernel
 *   kvw_mla_gather_latent              mla_prefill_branch_fp8 (latent copy)
 *   kvw_mla_gather_latent_fp8_dynamic  the same with dynamic FP8 scaling
 *   kvw_convert_bf16_to_fp8_e4m3       convert_bf16_to_fp8_e4m3fn
 *   kvw_quantize_fp8_rows              dynamic FP8 scaling, one scale per row
 *
 * Conventions shared by every call
 * --------------------------------
 * - Asynchronous: the call validates its host-side arguments, enqueues one
 *   kernel on `stream` and returns.  It never synchronises, never allocates
 *   device or host memory and keeps no state between calls.
 * - Ownership: every pointer is owned by the caller.  Pointers documented as
 *   "device" must be device-accessible (cudaMalloc / torch CUDA tensors) and
 *   stay valid until the kernel has finished; "host" pointers are read
 *   before the call returns.
 * - Element types are given by the KVW_DTYPE_* codes below; bf16 values are
 *   IEEE bfloat16, FP8 values OCP E4M3FN.
 * - Return value: KVW_OK, or an error code for argument errors found on the
 *   host (nothing is launched then), or KVW_ECUDA when the launch failed.
 * - Data errors found on the device (bad page ids, positions past the RoPE
 *   table, malformed offsets) do not abort: the affected rows are skipped
 *   and the matching KVW_ERR_* bit is OR-ed into *err_flags (a device
 *   uint32, optional: pass NULL to ignore).  The library only sets bits;
 *   zero the word before the call and read it after synchronising.
 *     KVW_ERR_PAGE     a slot maps to no valid page (page index >= the
 *                      table width, or page id >= num_pages, including the
 *                      0xFFFFFFFF "unmapped" sentinel): that cache row is not
 *                      written (query rows of the token still are);
 *     KVW_ERR_POSITION a RoPE position >= freqs_rows: nothing of that token
 *                      is written;
 *     KVW_ERR_OFFSETS  input_row_offsets does not start at 0, does not end
 *                      at the token count, or decreases: nothing is written.
 *     KVW_ERR_TIMEOUT  an internal pipeline wait (between the copy engine
 *                      and the compute warps of the GQA kernel or of the
 *                      dynamic-FP8 latent gather) gave up after about one
 *                      second of GPU time; the output is incomplete.  Reported instead of hanging
 *                      the GPU.  It is not expected on a healthy device, but
 *                      a CTA that the GPU pre-empts for longer than the
 *                      limit (time slicing with other processes on a shared
 *                      GPU) can report it spuriously.  With err_flags NULL
 *                      a timeout goes unnoticed: pass a flag word wherever
 *                      incomplete output must be detected.
 *   With zero tokens nothing is launched and nothing is checked.
 * - Ragged batches: input_row_offsets (device, uint32 [num_batches + 1])
 *   marks request boundaries in the flattened token dimension; request b
 *   owns tokens offsets[b] .. offsets[b+1]-1.  New token i of request b is
 *   written to cache slot position cache_lengths[b] + i, i.e. row
 *   (position % page_size) of page page_table[b][position / page_size].
 *   num_batches <= KVW_MAX_BATCHES.
 * - Alignment: every vector-accessed device pointer must be 16-byte
 *   aligned, and every row/head stride must keep rows 16-byte aligned
 *   (KVW_EINVAL otherwise).
 * - Aliasing: rows of different tokens must map to different cache slots
 *   (page tables hold distinct pages); otherwise the result is undefined.
 * - Size limits (KVW_EUNSUPPORTED beyond them): num_batches <= 8192; MLA
 *   tot_seq_len * num_heads * 8 <= 0xFFFFF000 (16-byte q vectors); GQA
 *   head_size a multiple of 16 and <= 512, and (num_q_heads + num_heads) *
 *   head_size / 16 <= 1024; K-norm gamma_len <= 2048 and normalised rows
 *   (tokens x heads) <= 0xFFFFF000.
 */
#ifndef KVW_H
#define KVW_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum kvw_status {
    KVW_OK = 0,
    KVW_EINVAL = 1,       /* bad argument (null, size, alignment, range) */
    KVW_EUNSUPPORTED = 2, /* valid but not implemented (dtype, shape) */
    KVW_ECUDA = 3         /* kernel launch failed */
};

enum kvw_dtype { KVW_DTYPE_BF16 = 0, KVW_DTYPE_FP8_E4M3 = 1, KVW_DTYPE_F32 = 2 };

enum kvw_err_bits {
    KVW_ERR_PAGE = 1u,
    KVW_ERR_POSITION = 2u,
    KVW_ERR_OFFSETS = 4u,
    KVW_ERR_TIMEOUT = 8u
};

#define KVW_MAX_BATCHES 8192u
#define KVW_PAGE_UNMAPPED 0xFFFFFFFFu

/*
 * Paged cache of one model ("PagedKVCacheCollection" / "KVCollectionT" on
 * the pages, which leave its layout open; this descriptor is our own).
 *
 * Element (page, kv, layer, row, head, col) lives at
 *   data + page*stride_page + kv*stride_kv + layer*stride_layer
 *        + row*stride_token + head*stride_head + col
 * in elements of `dtype`.  kv = 0 is K (the only plane the MLA latent cache
 * has); kv = 1 is V and is never touched.  The dense default layout is
 * [num_pages, kv, num_layers, page_size, num_heads, head_size].
 *
 *   data           device, the cache storage (read and written)
 *   dtype          KVW_DTYPE_BF16 or KVW_DTYPE_FP8_E4M3
 *   scale          FP8 dequantisation scale: a value y is stored as
 *                  satfinite_round_nearest_even(y / scale) (1.0 = no scaling)
 *   page_table     device, uint32 [num_batches, max_pages_per_seq]
 *   cache_lengths  device, uint32 [num_batches]: tokens already cached per
 *                  request before this step
 */
typedef struct kvw_paged_cache {
    void* data;
    int32_t dtype;
    float scale;
    const uint32_t* page_table;
    uint32_t max_pages_per_seq;
    const uint32_t* cache_lengths;
    uint32_t num_pages;
    uint32_t num_layers;
    uint32_t page_size;
    uint32_t num_heads;
    uint32_t head_size;
    int64_t stride_page;
    int64_t stride_kv;
    int64_t stride_layer;
    int64_t stride_token;
    int64_t stride_head;
} kvw_paged_cache_t;

/*
 * Fused MLA key-cache write ("mla_fused_rope_rmsnorm_quantization" page,
 * description and Args; "mla_graph" module page, entry
 * fused_rope_rmsnorm_quantization_kernel).  For every new token t at slot
 * position pos:
 *   q_rope_out[t, h, :] = RoPE(q_rope[t, h, :], freqs_cis[pos])   all heads h
 *   row = kv_in[t, 0:576]
 *   y[0:512]   = RMSNorm(row[0:512]) * gamma  (eps = epsilon, fp32)
 *   y[512:576] = RoPE(row[512:576], freqs_cis[pos])
 *   cache[page(pos), K, layer_idx, pos % page_size, 0, 0:576] = quant(y)
 * RoPE rotates adjacent pairs (2k, 2k+1) by freqs_cis[pos][2k] (cosine) and
 * freqs_cis[pos][2k+1] (sine).  quant is bf16 round-to-nearest-even, or the
 * FP8 rule of the descriptor's scale.
 *
 *   q_rope_out     device, [tot_seq_len, num_heads, 64], out_dtype: bf16, or
 *                  FP8 E4M3 by direct saturating conversion (no scale; the
 *                  out_rope_dtype parameter of the page)
 *   q_rope         device, bf16 [tot_seq_len, num_heads, 64], contiguous
 *   input_row_offsets, num_batches   ragged boundaries (see above)
 *   tot_seq_len    host-known number of new tokens (= offsets[num_batches])
 *   freqs_cis      device, freq_dtype (f32) [freqs_rows, 64]
 *   gamma          device, gamma_dtype (bf16) [512]
 *   kv_in          device, bf16 rows of 576 values (512 latent then 64 rope),
 *                  row t at kv_in + t*kv_row_stride elements (stride >= 576,
 *                  multiple of 8)
 *   cache          host pointer to the descriptor: num_heads 1, head_size
 *                  576, dtype bf16 or FP8 E4M3
 *   layer_idx      < cache->num_layers
 *   epsilon        RMSNorm epsilon
 * num_heads may be 0 (cache write only).
 */
int kvw_mla_rope_rmsnorm_quant(void* q_rope_out, int32_t out_dtype, const void* q_rope,
                               const uint32_t* input_row_offsets, uint32_t num_batches,
                               uint32_t tot_seq_len, uint32_t num_heads, const void* freqs_cis,
                               int32_t freq_dtype, uint32_t freqs_rows, const void* gamma,
                               int32_t gamma_dtype, const void* kv_in, int64_t kv_row_stride,
                               const kvw_paged_cache_t* cache, uint32_t layer_idx, float epsilon,
                               uint32_t* err_flags, cudaStream_t stream);

/*
 * In-place variant ("mla_graph" module page, entry fused_rope_rmsnorm_kernel;
 * the first two steps of the MLA decode and prefill branches): identical to
 * kvw_mla_rope_rmsnorm_quant except that each new token's 576-wide latent
 * row is read from its cache slot (written there by the latent projection)
 * and the normalised / rotated row is written back to the same slot.  A bf16
 * cache is read and written as bf16; an FP8 E4M3 cache is dequantised with
 * its scale, and re-quantised after.  Arguments as above without kv_in.
 */
int kvw_mla_rope_rmsnorm_inplace(void* q_rope_out, int32_t out_dtype, const void* q_rope,
                                 const uint32_t* input_row_offsets, uint32_t num_batches,
                                 uint32_t tot_seq_len, uint32_t num_heads, const void* freqs_cis,
                                 int32_t freq_dtype, uint32_t freqs_rows, const void* gamma,
                                 int32_t gamma_dtype, const kvw_paged_cache_t* cache,
                                 uint32_t layer_idx, float epsilon, uint32_t* err_flags,
                                 cudaStream_t stream);

/*
 * Paged -> contiguous copy of the MLA latent cache ("mla_graph" module page,
 * entry mla_prefill_branch_fp8: the KV latent values are copied out of the
 * paged cache into a contiguous buffer and quantised).  Request b's context
 * (cache positions 0 .. ctx_offsets[b+1] - ctx_offsets[b] - 1, i.e. prior plus
 * new tokens) is copied to out rows ctx_offsets[b] .. ctx_offsets[b+1] - 1.
 * Values are read as the cache holds them (bf16, or E4M3 times the cache
 * scale) and written as out_dtype: bf16 (round to nearest even) or FP8 E4M3
 * satfinite_round_nearest_even(v / out_scale).
 *
 *   out            device, [total_rows, 576] of out_dtype, 16-byte aligned
 *   cache          host pointer to the descriptor (num_heads 1, head_size 576)
 *   ctx_offsets    device, uint32 [num_batches + 1]: 0, non-decreasing, ending
 *                  at total_rows (else KVW_ERR_OFFSETS and nothing is written)
 * A row whose slot has no valid page is not written (KVW_ERR_PAGE).
 */
int kvw_mla_gather_latent(void* out, int32_t out_dtype, float out_scale,
                          const kvw_paged_cache_t* cache, uint32_t layer_idx,
                          const uint32_t* ctx_offsets, uint32_t num_batches, uint32_t total_rows,
                          uint32_t* err_flags, cudaStream_t stream);

/*
 * The same copy quantised with dynamic FP8 scaling, one scale per row (the
 * "mla_graph" module page: entry mla_prefill_branch_fp8 copies the KV latent
 * values out of the paged cache and quantises them to FP8; the module
 * description names dynamic FP8 scaling).  For each context row r, with v
 * its 576 values as the cache holds them (bf16, or E4M3 times the cache
 * scale):
 *   out_scales[r] = max_j |v_j| / 448   (1 for an all-zero row)
 *   out_codes[r][j] = satfinite_round_nearest_even(v_j / out_scales[r])
 * One pass over the cache: equal, codes and scales, to kvw_mla_gather_latent
 * to bf16 followed by kvw_quantize_fp8_rows for a bf16 cache.
 *
 *   out_codes    device, uint8 [total_rows, 576], 16-byte aligned
 *   out_scales   device, f32 [total_rows]
 *   other arguments, flags and errors as kvw_mla_gather_latent; a row
 *   without a valid page is not written (neither codes nor scale).  The
 *   rows reach the compute warps through bounded pipeline waits, so this
 *   call can also report KVW_ERR_TIMEOUT (see the flags above).
 */
int kvw_mla_gather_latent_fp8_dynamic(void* out_codes, float* out_scales,
                                      const kvw_paged_cache_t* cache, uint32_t layer_idx,
                                      const uint32_t* ctx_offsets, uint32_t num_batches,
                                      uint32_t total_rows, uint32_t* err_flags,
                                      cudaStream_t stream);

/*
 * bf16 -> FP8 E4M3 ("mla_graph" module page, convert_bf16_to_fp8_e4m3fn):
 * out[i] = satfinite_round_nearest_even(in[i] / scale), n a multiple of 8.
 *   out  device, n bytes, 8-byte aligned;  in  device, n bf16, 16-byte aligned
 */
int kvw_convert_bf16_to_fp8_e4m3(void* out, const void* in, uint64_t n, float scale,
                                 cudaStream_t stream);

/*
 * Dynamic FP8 scaling per row ("mla_graph" module page: dynamic FP8 scaling
 * of the FP8 branches; per-token granularity): for each row r,
 *   out_scales[r] = max_j |in[r][j]| / 448   (1 for an all-zero row)
 *   out_codes[r][j] = satfinite_round_nearest_even(in[r][j] / out_scales[r])
 * so the row's largest magnitude becomes +-448 and in ~= code * scale.
 *   in          device, bf16 rows of `cols` values, row stride in_row_stride
 *               elements (multiple of 8, 16-byte aligned); cols a multiple of 8
 *   out_codes   device, uint8 rows, row stride out_row_stride (multiple of 8)
 *   out_scales  device, f32 [rows]
 */
int kvw_quantize_fp8_rows(void* out_codes, float* out_scales, const void* in, uint32_t rows,
                          uint32_t cols, int64_t in_row_stride, int64_t out_row_stride,
                          cudaStream_t stream);

/*
 * Fused GQA Q/K RoPE ("generic_fused_qk_rope_bshd_paged_ragged" page,
 * description, Parameters and Args).  For every new token t:
 *   output[t, h, :] = RoPE(q_proj[t, h, :])              all q heads h
 *   K[slot(t), g, :] = RoPE(K[slot(t), g, :]) in place   all kv heads g
 * Pairs are (2k, 2k+1) when interleaved != 0, else (k, k + head_size/2).
 * Pair k uses the cosine/sine at freqs_cis[p][2k], [2k+1], where p is
 *   - the slot position when position_ids is NULL;
 *   - position_ids[t] when mrope_section is NULL;
 *   - position_ids[r * tot_seq_len + t] otherwise, r = 0 for
 *     k < s0, 1 for k < s0 + s1, else 2 (s = mrope_section, counted in
 *     rotary pairs, s0 + s1 + s2 = head_size / 2).
 * The K row is always the one of the slot position.
 *
 * An FP8 E4M3 K cache (the collection's scale_dtype_ /
 * quantization_granularity_ parameters; here a per-tensor scale) is
 * dequantised (code value times scale, fp32), rotated, and stored again as
 * satfinite_round_nearest_even(y / scale).
 *
 *   q_proj         device, bf16 [tot_seq_len, num_q_heads, head_size]
 *   cache          host pointer to the descriptor: bf16 or FP8 E4M3 (scale
 *                  > 0), head_size a multiple of 16 and <= 512
 *   freqs_cis      device, f32 [freqs_rows, head_size]
 *   position_ids   device, uint32 [tot_seq_len] or [3, tot_seq_len], or NULL
 *   mrope_section  HOST, uint32 [3], or NULL
 *   output         device, bf16 like q_proj; may be q_proj itself
 */
int kvw_qk_rope_paged_ragged(const void* q_proj, const uint32_t* input_row_offsets,
                             uint32_t num_batches, uint32_t tot_seq_len, uint32_t num_q_heads,
                             const kvw_paged_cache_t* cache, const void* freqs_cis,
                             uint32_t freqs_rows, const uint32_t* position_ids, int interleaved,
                             const uint32_t* mrope_section, uint32_t layer_idx, void* output,
                             uint32_t* err_flags, cudaStream_t stream);

/*
 * In-place RMSNorm of new K-cache entries ("rms_norm_kv_cache_ragged_paged"
 * page).  For every new token (total_seq_len of them, known on the host)
 * and, with per_head_norm != 0, every kv head g, the first gamma_len values
 * x of the K row are replaced by
 *   y_j = x_j * rsqrt(mean(x^2) + epsilon) * (gamma_j + weight_offset)
 * computed in fp32 and rounded once to bf16 (multiply_before_cast != 0), or
 * with the normalised value rounded to bf16 before the multiply
 * (multiply_before_cast == 0).  Columns >= gamma_len are not touched.
 * The sum of squares is accumulated in an order of the kernel's choosing
 * and, for 8-aligned gamma lengths of contiguous rows, the 1/rms factor is
 * an rsqrt estimate refined by one Newton-Raphson step (within two fp32 ulp
 * of the correctly rounded value): results are within one bf16 ulp of a
 * correctly rounded evaluation of the formula (two roundings' worth with
 * multiply_before_cast == 0).
 * With per_head_norm == 0 the whole K row of the token (num_heads *
 * head_size values) is normalised as one vector and gamma_len must equal
 * that width.
 *
 *   cache          host pointer to the descriptor (bf16)
 *   gamma          device, bf16 [gamma_len]; 1 <= gamma_len <= head_size
 *                  (per-head), gamma_len <= 2048
 */
int kvw_rms_norm_kv_cache_paged(const kvw_paged_cache_t* cache, const void* gamma,
                                uint32_t gamma_len, float epsilon, float weight_offset,
                                uint32_t layer_idx, uint32_t total_seq_len,
                                const uint32_t* input_row_offsets, uint32_t num_batches,
                                int multiply_before_cast, int per_head_norm, uint32_t* err_flags,
                                cudaStream_t stream);

/* Name of a kvw_status value (static string). */
const char* kvw_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int kvw_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVW_H */
