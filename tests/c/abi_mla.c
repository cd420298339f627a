/*
 * The C ABI used from plain C: allocate device buffers, run the fused MLA
 * cache write on a small ragged batch (2 requests, new tokens [3, 5], prior
 * lengths [0, 7], 4 q heads, page size 16, layer 1 of 2), copy the results
 * back and compare them with the CPU reference on the same inputs: query
 * rows within 1 bf16 ulp, written cache rows within 1 bf16 ulp (bf16 cache)
 * or 1 E4M3 ulp on at most 0.1% of the written values (FP8 cache), every
 * other cache byte unchanged, equal error flags.
 *
 * Usage: abi_mla <cache dtype: 0 bf16 | 1 fp8>   (exit status 0 on success)
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kvw.h"

/* CPU reference (oracle/oracle.c), linked from liboracle.so */
uint32_t oracle_mla_rope_rmsnorm_quant(
    void* q_rope_out, int out_dtype, const uint16_t* q_rope, const uint32_t* offsets, uint32_t B,
    uint32_t T, uint32_t H, const float* freqs, uint32_t freqs_rows, const uint16_t* gamma,
    const uint16_t* kv_in, int64_t kv_row_stride, void* cache, int cache_dtype, float scale,
    const uint32_t* page_table, uint32_t max_pages, const uint32_t* cache_lengths,
    uint32_t num_pages, uint32_t num_layers, uint32_t page_size, uint32_t num_heads,
    uint32_t head_size, int64_t s_page, int64_t s_kv, int64_t s_layer, int64_t s_token,
    int64_t s_head, uint32_t layer_idx, float eps, int nthreads);
void oracle_bf16_encode(const float* x, uint16_t* out, int64_t n);

enum { B = 2, T = 8, H = 4, P = 16, PAGES = 8, LAYERS = 2, LAYER = 1, MAXP = 4, ROW = 576,
       ROWS = 64 };

static uint32_t lcg_state = 12345u;
static float uniform(float lo, float hi) { /* a fixed LCG: reproducible inputs */
    lcg_state = lcg_state * 1664525u + 1013904223u;
    return lo + (hi - lo) * (float)(lcg_state >> 8) / 16777216.0f;
}

static int bf16_ordinal(uint16_t h) { return (h & 0x8000) ? -(int)(h & 0x7fff) : (int)h; }
static int e4m3_ordinal(uint8_t c) { return (c & 0x80) ? -(int)(c & 0x7f) : (int)c; }

#define CHECK(call)                                                         \
    do {                                                                    \
        cudaError_t e_ = (call);                                            \
        if (e_ != cudaSuccess) {                                            \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));     \
            return 2;                                                       \
        }                                                                   \
    } while (0)

int main(int argc, char** argv) {
    const int fp8 = argc > 1 && atoi(argv[1]) == 1;
    const size_t esz = fp8 ? 1 : 2;
    const uint32_t offsets[B + 1] = {0, 3, 8}, clen[B] = {0, 7};
    const uint32_t table[B * MAXP] = {5, 2, 7, 0, 1, 6, 3, 4};
    const int64_t s_token = ROW, s_layer = (int64_t)P * ROW, s_kv = LAYERS * s_layer;
    const int64_t s_page = s_kv;  /* one plane: the latent cache has no V */
    const size_t n_cache = (size_t)PAGES * s_page;

    /* inputs */
    static float qf[T * H * 64], kvf[T * ROW], gf[512], freqs[ROWS * 64];
    static uint16_t q[T * H * 64], kv[T * ROW], gamma[512];
    for (int i = 0; i < T * H * 64; ++i) qf[i] = uniform(-2.0f, 2.0f);
    for (int i = 0; i < T * ROW; ++i) kvf[i] = uniform(-2.0f, 2.0f);
    for (int i = 0; i < 512; ++i) gf[i] = uniform(0.8f, 1.2f);
    oracle_bf16_encode(qf, q, T * H * 64);
    oracle_bf16_encode(kvf, kv, T * ROW);
    oracle_bf16_encode(gf, gamma, 512);
    for (int p = 0; p < ROWS; ++p)
        for (int k = 0; k < 32; ++k) {
            const double a = p * pow(10000.0, -2.0 * k / 64.0);
            freqs[p * 64 + 2 * k] = (float)cos(a);
            freqs[p * 64 + 2 * k + 1] = (float)sin(a);
        }
    unsigned char* cache0 = malloc(n_cache * esz);
    for (size_t i = 0; i < n_cache * esz; ++i) cache0[i] = (unsigned char)(uniform(0.0f, 256.0f));

    /* reference */
    unsigned char* cache_ref = malloc(n_cache * esz);
    memcpy(cache_ref, cache0, n_cache * esz);
    static uint16_t q_ref[T * H * 64];
    const uint32_t f_ref = oracle_mla_rope_rmsnorm_quant(
        q_ref, 0, q, offsets, B, T, H, freqs, ROWS, gamma, kv, ROW, cache_ref, fp8, 1.0f, table,
        MAXP, clen, PAGES, LAYERS, P, 1, ROW, s_page, s_kv, s_layer, s_token, ROW, LAYER, 1e-6f, 1);

    /* the library, through the C ABI */
    void *d_q, *d_qo, *d_kv, *d_g, *d_f, *d_c, *d_off, *d_cl, *d_pt, *d_err;
    CHECK(cudaMalloc(&d_q, sizeof q));
    CHECK(cudaMalloc(&d_qo, sizeof q));
    CHECK(cudaMalloc(&d_kv, sizeof kv));
    CHECK(cudaMalloc(&d_g, sizeof gamma));
    CHECK(cudaMalloc(&d_f, sizeof freqs));
    CHECK(cudaMalloc(&d_c, n_cache * esz));
    CHECK(cudaMalloc(&d_off, sizeof offsets));
    CHECK(cudaMalloc(&d_cl, sizeof clen));
    CHECK(cudaMalloc(&d_pt, sizeof table));
    CHECK(cudaMalloc(&d_err, 4));
    CHECK(cudaMemcpy(d_q, q, sizeof q, cudaMemcpyHostToDevice));
    CHECK(cudaMemset(d_qo, 0, sizeof q));
    CHECK(cudaMemcpy(d_kv, kv, sizeof kv, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_g, gamma, sizeof gamma, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_f, freqs, sizeof freqs, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_c, cache0, n_cache * esz, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_off, offsets, sizeof offsets, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_cl, clen, sizeof clen, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(d_pt, table, sizeof table, cudaMemcpyHostToDevice));
    CHECK(cudaMemset(d_err, 0, 4));
    kvw_paged_cache_t desc = {d_c, fp8 ? KVW_DTYPE_FP8_E4M3 : KVW_DTYPE_BF16, 1.0f,
                              (const uint32_t*)d_pt, MAXP, (const uint32_t*)d_cl, PAGES, LAYERS,
                              P, 1, ROW, s_page, s_kv, s_layer, s_token, ROW};
    const int st = kvw_mla_rope_rmsnorm_quant(
        d_qo, KVW_DTYPE_BF16, d_q, (const uint32_t*)d_off, B, T, H, d_f, KVW_DTYPE_F32, ROWS, d_g,
        KVW_DTYPE_BF16, d_kv, ROW, &desc, LAYER, 1e-6f, (uint32_t*)d_err, 0);
    if (st != KVW_OK) {
        fprintf(stderr, "kvw_mla_rope_rmsnorm_quant: %s\n", kvw_status_string(st));
        return 1;
    }
    CHECK(cudaDeviceSynchronize());
    static uint16_t q_gpu[T * H * 64];
    unsigned char* cache_gpu = malloc(n_cache * esz);
    uint32_t f_gpu = 0;
    CHECK(cudaMemcpy(q_gpu, d_qo, sizeof q_gpu, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(cache_gpu, d_c, n_cache * esz, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(&f_gpu, d_err, 4, cudaMemcpyDeviceToHost));

    /* compare */
    int bad = 0;
    if (f_gpu != f_ref) {
        fprintf(stderr, "flags %u vs %u\n", f_gpu, f_ref);
        ++bad;
    }
    for (int i = 0; i < T * H * 64; ++i)
        if (abs(bf16_ordinal(q_gpu[i]) - bf16_ordinal(q_ref[i])) > 1) ++bad;
    unsigned char* written = calloc(n_cache, 1);
    for (int b = 0; b < B; ++b)
        for (uint32_t t = offsets[b]; t < offsets[b + 1]; ++t) {
            const uint32_t pos = clen[b] + (t - offsets[b]);
            const int64_t base = (int64_t)table[b * MAXP + pos / P] * s_page + LAYER * s_layer +
                                 (int64_t)(pos % P) * s_token;
            memset(written + base, 1, ROW);
        }
    size_t n_written = 0, n_fp8_off = 0;
    for (size_t i = 0; i < n_cache; ++i) {
        int d;
        if (fp8)
            d = abs(e4m3_ordinal(cache_gpu[i]) - e4m3_ordinal(cache_ref[i]));
        else {
            uint16_t a, r;
            memcpy(&a, cache_gpu + 2 * i, 2);
            memcpy(&r, cache_ref + 2 * i, 2);
            d = abs(bf16_ordinal(a) - bf16_ordinal(r));
        }
        if (d > (written[i] ? 1 : 0)) ++bad;
        n_written += written[i];
        if (fp8 && written[i] && d == 1) ++n_fp8_off;
    }
    /* FP8: 1-ulp differences allowed on at most 0.1% of the written values */
    if (fp8 && (double)n_fp8_off > 1e-3 * (double)n_written) {
        fprintf(stderr, "fp8: %zu of %zu written values 1 ulp off\n", n_fp8_off, n_written);
        ++bad;
    }
    printf("kvw %d (%s cache): %d mismatches, flags %u\n", kvw_version(), fp8 ? "fp8" : "bf16",
           bad, f_gpu);
    return bad ? 1 : 0;
}
