// Paged -> contiguous copy of the MLA latent cache, with type conversion.
//
// Operation: the step of the FP8 MLA prefill branch that copies the KV latent
// values of each request's whole context from the paged cache into a
// contiguous buffer and quantises them ("mla_graph" module page, entry
// mla_prefill_branch_fp8; the copy feeds the K/V up-projection GEMMs).
//
// GB300 design: pure streaming with persistent CTAs (one wave, the occupancy
// the register count allows).  A CTA stages the context offsets once, then
// walks tiles of kTileRows consecutive output rows.  A tile is 32 x 72
// pieces of 8 values; each of the 256 threads moves the same 9 pieces of
// every tile (fixed row and column slots), so all lanes stay busy and the 9
// loads of a thread are in flight together.  The cache address of each row
// of a tile (request by binary search over the staged offsets, page from the
// page table) is resolved by the first 32 threads one tile ahead, into the
// other half of a double-buffered shared array, while the current tile's
// loads are in flight; consecutive rows of one page are adjacent in memory,
// so a tile's loads are mostly one contiguous run.
#include <cstdint>

#include "kvw_device.cuh"

namespace kvw {
namespace {

constexpr uint32_t kThreads = 256;
constexpr uint32_t kRow = 576;
constexpr uint32_t kPiecesPerRow = kRow / 8;                                 // 72
constexpr uint32_t kTileRows = 32;
constexpr uint32_t kPiecesPerThread = kTileRows * kPiecesPerRow / kThreads;  // 9
static_assert(kTileRows * kPiecesPerRow == kPiecesPerThread * kThreads, "tile shape");

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

// Raw bytes of 8 cache elements at element offset `e` (16 bytes of bf16 or
// 8 bytes of E4M3, kept in .x/.y).
template <bool CF8>
__device__ __forceinline__ uint4 load_raw8(const unsigned char* cache, int64_t e) {
    if (CF8) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(cache + e));
        return make_uint4(v.x, v.y, 0, 0);
    }
    return ld_stream(reinterpret_cast<const uint4*>(cache + e * 2));
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

// Cache element offset of output row r (or -1: no valid page, flagged).
__device__ __forceinline__ int64_t row_base(const GatherArgs& a, const uint32_t* s_off,
                                            uint32_t r) {
    if (r >= a.rows) return -1;
    const uint32_t b = find_request(s_off, a.B, r);
    const uint32_t pos = r - s_off[b];
    const uint32_t pidx = pos / a.page_size;
    const uint32_t page = pidx < a.max_pages
                              ? __ldg(a.page_table + (uint64_t)b * a.max_pages + pidx)
                              : KVW_PAGE_UNMAPPED;
    if (page >= a.num_pages) {
        flag(a.err_flags, KVW_ERR_PAGE);
        return -1;
    }
    return (int64_t)page * a.s_page + a.layer_off + (int64_t)(pos - pidx * a.page_size) * a.s_token;
}

template <bool CF8, bool OF8>
__global__ void __launch_bounds__(kThreads, 4) gather_kernel(const GatherArgs a) {
    __shared__ int64_t s_base[2][kTileRows];
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
    const uint32_t tiles = (a.rows + kTileRows - 1) / kTileRows;
    uint32_t tile = blockIdx.x;
    if (tile >= tiles) return;
    if (threadIdx.x < kTileRows) s_base[0][threadIdx.x] = row_base(a, s_off, tile * kTileRows + threadIdx.x);
    __syncthreads();
    // this thread's fixed pieces: (row slot, column) of piece threadIdx.x + k * kThreads
    uint32_t prow[kPiecesPerThread], pcol[kPiecesPerThread];
#pragma unroll
    for (uint32_t k = 0; k < kPiecesPerThread; ++k) {
        const uint32_t p = threadIdx.x + k * kThreads;
        prow[k] = p / kPiecesPerRow;
        pcol[k] = (p % kPiecesPerRow) * 8;
    }
    uint32_t buf = 0;
    for (; tile < tiles; tile += gridDim.x, buf ^= 1u) {
        uint4 raw[kPiecesPerThread];
#pragma unroll
        for (uint32_t k = 0; k < kPiecesPerThread; ++k) {
            const int64_t base = s_base[buf][prow[k]];
            if (base >= 0) raw[k] = load_raw8<CF8>(a.cache, base + pcol[k]);
        }
        const uint32_t next = tile + gridDim.x;
        if (next < tiles && threadIdx.x < kTileRows)
            s_base[buf ^ 1u][threadIdx.x] = row_base(a, s_off, next * kTileRows + threadIdx.x);
#pragma unroll
        for (uint32_t k = 0; k < kPiecesPerThread; ++k) {
            if (s_base[buf][prow[k]] < 0) continue;
            float v[8];
            to_f32<CF8>(raw[k], a.cache_scale, v);
            const uint64_t e = (uint64_t)(tile * kTileRows + prow[k]) * kRow + pcol[k];
            store_k8<OF8>(a.out + e * (OF8 ? 1 : 2), v, a.out_scale);
        }
        __syncthreads();  // next tile's bases visible; this tile's no longer read
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
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem);
    if (e != cudaSuccess) return e;
    const uint32_t tiles = (a.rows + kTileRows - 1) / kTileRows;
    const uint32_t wave = (uint32_t)(sms * (per_sm > 0 ? per_sm : 1));
    k<<<tiles < wave ? tiles : wave, kThreads, smem, stream>>>(a);
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
