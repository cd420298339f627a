// Paged -> contiguous copy of the MLA latent cache, with type conversion.
//
// Operation: the step of the FP8 MLA prefill branch that copies the KV latent
// values of each request's whole context from the paged cache into a
// contiguous buffer and quantises them ("mla_graph" module page, entry
// mla_prefill_branch_fp8; the copy feeds the K/V up-projection GEMMs).
//
// GB300 design: pure streaming.  One warp per output row (576 values): the
// row's request comes from a binary search over the context offsets staged in
// shared memory, its page from the page table; lanes move 16-byte (bf16) or
// 8-byte (E4M3) pieces, convert in registers and store.  Each warp handles
// kRowsPerWarp rows with all loads issued before any store.
#include <cstdint>

#include "kvw_device.cuh"

namespace kvw {
namespace {

constexpr uint32_t kThreads = 256;
constexpr uint32_t kRowsPerWarp = 4;
constexpr uint32_t kRow = 576;

struct GatherArgs {
    unsigned char* out;
    const unsigned char* cache;
    const uint32_t* ctx_offsets;
    const uint32_t* page_table;
    uint32_t* err_flags;
    int64_t s_page, s_token, layer_off;  // cache elements
    uint32_t B, rows, max_pages, num_pages, page_size;
    float cache_scale, out_scale;
};

// Raw bytes of 8 cache elements starting at element `col` (16 bytes of bf16
// or 8 bytes of E4M3, kept in .x/.y).
template <bool CF8>
__device__ __forceinline__ uint4 load_raw8(const GatherArgs& a, int64_t base, uint32_t col) {
    if (CF8) {
        const uint2 v = *reinterpret_cast<const uint2*>(a.cache + base + col);
        return make_uint4(v.x, v.y, 0, 0);
    }
    return *reinterpret_cast<const uint4*>(a.cache + (base + col) * 2);
}

// Raw cache elements -> fp32 values (E4M3 times the cache scale).
template <bool CF8>
__device__ __forceinline__ void to_f32(const uint4& raw, float scale, float (&f)[8]) {
    if (CF8) {
        unpack8_e4m3(make_uint2(raw.x, raw.y), f);
        if (scale != 1.0f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], scale);
        }
    } else {
        unpack8(raw, f);
    }
}

template <bool CF8, bool OF8>
__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherArgs a) {
    extern __shared__ uint32_t s_off[];
    int ok = 1;
    for (uint32_t i = threadIdx.x; i <= a.B; i += blockDim.x) {
        const uint32_t o = __ldg(a.ctx_offsets + i);
        s_off[i] = o;
        if (i < a.B && o > __ldg(a.ctx_offsets + i + 1)) ok = 0;
        if ((i == 0 && o != 0u) || (i == a.B && o != a.rows)) ok = 0;
    }
    if (!__syncthreads_and(ok)) {
        if (threadIdx.x == 0) flag(a.err_flags, KVW_ERR_OFFSETS);
        return;
    }
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t warp_global = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const uint32_t r0 = warp_global * kRowsPerWarp;
    // lane l owns columns 8l..8l+7, 256+8l.., and (l < 8) 512+8l..
    int64_t base[kRowsPerWarp];
    uint4 raw[kRowsPerWarp][3];
#pragma unroll
    for (uint32_t q = 0; q < kRowsPerWarp; ++q) {
        const uint32_t r = r0 + q;
        base[q] = -1;
        if (r < a.rows) {
            const uint32_t b = find_request(s_off, a.B, r);
            const uint32_t pos = r - s_off[b];
            const uint32_t pidx = pos / a.page_size;
            const uint32_t page =
                pidx < a.max_pages ? __ldg(a.page_table + (uint64_t)b * a.max_pages + pidx)
                                   : KVW_PAGE_UNMAPPED;
            if (page < a.num_pages)
                base[q] = (int64_t)page * a.s_page + a.layer_off +
                          (int64_t)(pos - pidx * a.page_size) * a.s_token;
            else if (lane == 0)
                flag(a.err_flags, KVW_ERR_PAGE);
        }
        if (base[q] >= 0) {
            raw[q][0] = load_raw8<CF8>(a, base[q], lane * 8);
            raw[q][1] = load_raw8<CF8>(a, base[q], 256 + lane * 8);
            if (lane < 8) raw[q][2] = load_raw8<CF8>(a, base[q], 512 + lane * 8);
        }
    }
#pragma unroll
    for (uint32_t q = 0; q < kRowsPerWarp; ++q) {
        if (base[q] < 0) continue;
        unsigned char* orow = a.out + (uint64_t)(r0 + q) * kRow * (OF8 ? 1 : 2);
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            if (j == 2 && lane >= 8) break;
            const uint32_t col = 256u * j + lane * 8;
            float v[8];
            to_f32<CF8>(raw[q][j], a.cache_scale, v);
            store_k8<OF8>(orow + col * (OF8 ? 1 : 2), v, a.out_scale);
        }
    }
}

template <bool CF8, bool OF8>
cudaError_t launch(const GatherArgs& a, cudaStream_t stream) {
    auto k = gather_kernel<CF8, OF8>;
    const size_t smem = sizeof(uint32_t) * ((size_t)a.B + 1);
    if (smem > 32 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const uint32_t rows_per_cta = (kThreads / 32) * kRowsPerWarp;
    k<<<(a.rows + rows_per_cta - 1) / rows_per_cta, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvw

extern "C" int kvw_mla_gather_latent(void* out, int32_t out_dtype, float out_scale,
                                     const kvw_paged_cache_t* cache, uint32_t layer_idx,
                                     const uint32_t* ctx_offsets, uint32_t num_batches,
                                     uint32_t total_rows, uint32_t* err_flags,
                                     cudaStream_t stream) {
    using namespace kvw;
    if (!cache) return KVW_EINVAL;
    if (out_dtype != KVW_DTYPE_BF16 && out_dtype != KVW_DTYPE_FP8_E4M3) return KVW_EUNSUPPORTED;
    if (cache->dtype != KVW_DTYPE_BF16 && cache->dtype != KVW_DTYPE_FP8_E4M3) return KVW_EUNSUPPORTED;
    if (cache->head_size != kRow || cache->num_heads != 1) return KVW_EUNSUPPORTED;
    if (num_batches > KVW_MAX_BATCHES) return KVW_EUNSUPPORTED;
    if (total_rows == 0) return KVW_OK;
    const bool cf8 = cache->dtype == KVW_DTYPE_FP8_E4M3, of8 = out_dtype == KVW_DTYPE_FP8_E4M3;
    const int64_t esz = cf8 ? 1 : 2;
    if (!out || !ctx_offsets || !cache->data || !cache->page_table) return KVW_EINVAL;
    if (layer_idx >= cache->num_layers || cache->page_size == 0 || cache->max_pages_per_seq == 0)
        return KVW_EINVAL;
    if ((cf8 && !(cache->scale > 0.0f && cache->scale < 3.0e38f)) ||
        (of8 && !(out_scale > 0.0f && out_scale < 3.0e38f)))
        return KVW_EINVAL;
    if (!aligned16(out) || !aligned16(cache->data)) return KVW_EINVAL;
    if ((cache->stride_page * esz) % 16 || (cache->stride_layer * esz) % 16 ||
        (cache->stride_token * esz) % 16 || cache->stride_page <= 0 || cache->stride_token <= 0)
        return KVW_EINVAL;
    GatherArgs a;
    a.out = static_cast<unsigned char*>(out);
    a.cache = static_cast<const unsigned char*>(cache->data);
    a.ctx_offsets = ctx_offsets;
    a.page_table = cache->page_table;
    a.err_flags = err_flags;
    a.s_page = cache->stride_page;
    a.s_token = cache->stride_token;
    a.layer_off = (int64_t)layer_idx * cache->stride_layer;
    a.B = num_batches;
    a.rows = total_rows;
    a.max_pages = cache->max_pages_per_seq;
    a.num_pages = cache->num_pages;
    a.page_size = cache->page_size;
    a.cache_scale = cache->scale;
    a.out_scale = out_scale;
    const cudaError_t e = cf8 ? (of8 ? launch<true, true>(a, stream) : launch<true, false>(a, stream))
                              : (of8 ? launch<false, true>(a, stream) : launch<false, false>(a, stream));
    return e == cudaSuccess ? KVW_OK : KVW_ECUDA;
}
