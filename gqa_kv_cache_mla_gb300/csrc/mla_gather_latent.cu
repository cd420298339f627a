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
    FastDiv ps_div;  // division by page_size
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
    const uint32_t pidx = fast_div(pos, a.ps_div);
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

// Copy with dynamic per-row FP8.  A row's scale needs all of its 576 values,
// so here a warp owns whole rows, kDynRows at a time (lane l holds pieces l
// and l + 32 of each, and the tail piece l % 8 of row l / 8): the row maxima
// are integer maxima of bit patterns and one warp redux per row,
// the scale and its reciprocal are computed in registers and every piece is
// quantised from the registers that still hold it -- no shared-memory
// reduction and no block barrier after the offsets are staged.  Warps are
// persistent; lane q < kDynRows resolves the page of row q of the warp's next
// step while the current step's loads are in flight.  Values that are bf16
// numbers (a bf16 cache, or E4M3 codes at cache scale 1) divide by the scale
// through div_refined; others through the IEEE divide.
constexpr uint32_t kDynRows = 4;

// base[i] for a run-time i < kDynRows, without indexing registers dynamically
__device__ __forceinline__ int64_t base_of(const int64_t (&base)[kDynRows], uint32_t i) {
    int64_t b = base[0];
#pragma unroll
    for (uint32_t q = 1; q < kDynRows; ++q) b = i == q ? base[q] : b;
    return b;
}

// Bit pattern of the largest magnitude among 8 cache values, as an fp32
// (non-negative floats order like their bit patterns).  bf16: the patterns
// with the sign cleared order like the magnitudes, so a per-halfword
// unsigned max finds it; E4M3 codes likewise per byte.  A NaN (a pattern
// above infinity, or code 0x7F) falls back to the float maximum, which
// ignores it, as the reference maximum does.
template <bool CF8>
__device__ __forceinline__ uint32_t piece_max_bits(const uint4& raw, float cache_scale) {
    if (!CF8) {
        const uint32_t acc = __vmaxu2(__vmaxu2(raw.x & 0x7fff7fffu, raw.y & 0x7fff7fffu),
                                      __vmaxu2(raw.z & 0x7fff7fffu, raw.w & 0x7fff7fffu));
        const uint32_t m = max(acc & 0xffffu, acc >> 16);
        if (m <= 0x7f80u) return m << 16;
    } else {
        const uint32_t acc = __vmaxu4(raw.x & 0x7f7f7f7fu, raw.y & 0x7f7f7f7fu);
        const uint32_t m = max(max(acc & 0xffu, (acc >> 8) & 0xffu), max((acc >> 16) & 0xffu, acc >> 24));
        if (m != 0x7fu) {
            const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(m), __NV_E4M3);
            const float f = __half2float(__half(h));
            return __float_as_uint(cache_scale == 1.0f ? f : __fmul_rn(f, cache_scale));
        }
    }
    float v[8];
    to_f32<CF8>(raw, cache_scale, v);
    float f = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) f = fmaxf(f, fabsf(v[e]));
    return __float_as_uint(f);
}

// Per-halfword maxima of the sign-cleared bf16 patterns of a piece, merged
// into acc (bf16 magnitudes order like their patterns).
__device__ __forceinline__ uint32_t halves_max(uint32_t acc, const uint4& raw) {
    return __vmaxu2(acc, __vmaxu2(__vmaxu2(raw.x & 0x7fff7fffu, raw.y & 0x7fff7fffu),
                                  __vmaxu2(raw.z & 0x7fff7fffu, raw.w & 0x7fff7fffu)));
}

// 8 cache values -> 8 E4M3 codes of value / sc (y = RN(1/sc); see div_refined).
template <bool CF8>
__device__ __forceinline__ uint2 quantize_piece(const uint4& raw, float cache_scale, float sc,
                                                float y, bool fast) {
    float v[8];
    to_f32<CF8>(raw, cache_scale, v);
    if (!CF8 && fast) {
        // magnitudes divided on fp32 pairs, codes of the magnitudes, then the
        // bf16 sign bits (byte 1 and 3 of each word) or-ed into the code bytes
        const float2 ns2 = make_float2(-sc, -sc), y2 = make_float2(y, y);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float2 x2 = make_float2(fabsf(v[e]), fabsf(v[e + 1]));
            const float2 q0 = __fmul2_rn(x2, y2);
            const float2 r = __ffma2_rn(q0, ns2, x2);
            const float2 q = __ffma2_rn(r, y2, q0);
            v[e] = q.x;
            v[e + 1] = q.y;
        }
        uint2 c = pack8_e4m3(v);
        c.x |= __byte_perm(raw.x, raw.y, 0x7531u) & 0x80808080u;
        c.y |= __byte_perm(raw.z, raw.w, 0x7531u) & 0x80808080u;
        return c;
    }
    if (fast) {
        // div_refined on fp32 pairs: the packed multiply and fused
        // multiply-add round each component exactly as the scalar ones, and
        // x - q0 s is formed as fma(q0, -s, x)
        const float2 ns2 = make_float2(-sc, -sc), y2 = make_float2(y, y);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float2 x2 = make_float2(v[e], v[e + 1]);
            const float2 q0 = __fmul2_rn(x2, y2);
            const float2 r = __ffma2_rn(q0, ns2, x2);
            const float2 q = __ffma2_rn(r, y2, q0);
            v[e] = copysignf(q.x, x2.x);
            v[e + 1] = copysignf(q.y, x2.y);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __fdiv_rn(v[e], sc);
    }
    return pack8_e4m3(v);
}

template <bool CF8>
__global__ void __launch_bounds__(kThreads, 3) gather_dynamic_kernel(const GatherArgs a,
                                                                     float* scales) {
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
    const uint32_t nwarps = gridDim.x * (kThreads / 32);
    const uint32_t steps = (a.rows + kDynRows - 1) / kDynRows;
    uint32_t st = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    int64_t base_lane = (st < steps && lane < kDynRows) ? row_base(a, s_off, st * kDynRows + lane)
                                                         : -1;
    const bool bf16_values = !CF8 || a.cache_scale == 1.0f;
    // lane l also moves the tail piece (columns 512 + 8 (l & 7) ..) of row
    // l / 8, so every lane moves 9 pieces per step
    const uint32_t tq = lane >> 3, tcol = 512u + 8u * (lane & 7u);
    for (; st < steps; st += nwarps) {
        int64_t base[kDynRows];
        uint4 raw[kDynRows][2], rtail;
#pragma unroll
        for (uint32_t q = 0; q < kDynRows; ++q) {
            base[q] = __shfl_sync(0xffffffffu, base_lane, q);
            if (base[q] >= 0) {
                raw[q][0] = load_raw8<CF8>(a.cache, base[q] + lane * 8);
                raw[q][1] = load_raw8<CF8>(a.cache, base[q] + 256 + lane * 8);
            }
        }
        const int64_t btail = base_of(base, tq);
        if (btail >= 0) rtail = load_raw8<CF8>(a.cache, btail + tcol);
        const uint32_t next = st + nwarps;
        base_lane = (next < steps && lane < kDynRows) ? row_base(a, s_off, next * kDynRows + lane)
                                                      : -1;
        // row maxima as bit patterns of non-negative floats (which order like
        // the values): per lane, then one redux over the warp per row
        uint32_t mbits[kDynRows];
        if constexpr (!CF8) {
            const uint32_t atail = btail >= 0 ? halves_max(0u, rtail) : 0u;
#pragma unroll
            for (uint32_t q = 0; q < kDynRows; ++q) {
                uint32_t acc = tq == q ? atail : 0u;
                if (base[q] >= 0) acc = halves_max(halves_max(acc, raw[q][0]), raw[q][1]);
                uint32_t mq = max(acc & 0xffffu, acc >> 16);
                if (mq > 0x7f80u) {  // a NaN among this lane's values of row q: float maximum
                    float f = 0.0f;
                    if (base[q] >= 0) f = fmaxf(__uint_as_float(piece_max_bits<CF8>(raw[q][0], 1.0f)),
                                                __uint_as_float(piece_max_bits<CF8>(raw[q][1], 1.0f)));
                    if (tq == q && btail >= 0)
                        f = fmaxf(f, __uint_as_float(piece_max_bits<CF8>(rtail, 1.0f)));
                    mq = __float_as_uint(f);
                } else {
                    mq <<= 16;
                }
                mbits[q] = __reduce_max_sync(0xffffffffu, mq);
            }
        } else {
            uint32_t mtail = btail >= 0 ? piece_max_bits<CF8>(rtail, a.cache_scale) : 0u;
#pragma unroll
            for (uint32_t q = 0; q < kDynRows; ++q) {
                uint32_t mq = tq == q ? mtail : 0u;
                if (base[q] >= 0) {
                    mq = max(mq, piece_max_bits<CF8>(raw[q][0], a.cache_scale));
                    mq = max(mq, piece_max_bits<CF8>(raw[q][1], a.cache_scale));
                }
                mbits[q] = __reduce_max_sync(0xffffffffu, mq);
            }
        }
        // lane q turns row q's maximum into its scale and reciprocal
        uint32_t mine = mbits[0];
#pragma unroll
        for (uint32_t q = 1; q < kDynRows; ++q) mine = lane == q ? mbits[q] : mine;
        const float amax = __uint_as_float(mine);
        const float sc_lane = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        const float y_lane = __frcp_rn(sc_lane);
        if (lane < kDynRows && base_of(base, lane) >= 0)
            scales[(uint64_t)st * kDynRows + lane] = sc_lane;
        float sc[kDynRows], y[kDynRows];
#pragma unroll
        for (uint32_t q = 0; q < kDynRows; ++q) {
            sc[q] = __shfl_sync(0xffffffffu, sc_lane, q);
            y[q] = __shfl_sync(0xffffffffu, y_lane, q);
        }
#pragma unroll
        for (uint32_t q = 0; q < kDynRows; ++q) {
            if (base[q] < 0) continue;  // warp-uniform
            const uint64_t r = (uint64_t)st * kDynRows + q;
            const bool fast = bf16_values && refined_ok(sc[q]);
#pragma unroll
            for (uint32_t j = 0; j < 2; ++j)
                *reinterpret_cast<uint2*>(a.out + r * kRow + 256u * j + lane * 8) =
                    quantize_piece<CF8>(raw[q][j], a.cache_scale, sc[q], y[q], fast);
        }
        if (btail >= 0) {
            float st_ = sc[0], yt = y[0];
#pragma unroll
            for (uint32_t q = 1; q < kDynRows; ++q) {
                st_ = tq == q ? sc[q] : st_;
                yt = tq == q ? y[q] : yt;
            }
            const uint64_t r = (uint64_t)st * kDynRows + tq;
            *reinterpret_cast<uint2*>(a.out + r * kRow + tcol) =
                quantize_piece<CF8>(rtail, a.cache_scale, st_, yt, bf16_values && refined_ok(st_));
        }
    }
}

template <bool CF8, bool OF8>
cudaError_t launch(const GatherArgs& a, cudaStream_t stream) {
    constexpr auto k = gather_kernel<CF8, OF8>;
    const size_t smem = sizeof(uint32_t) * ((size_t)a.B + 1);
    uint64_t wave = 0;
    const cudaError_t e = wave_ctas<k>(kThreads, smem, wave);
    if (e != cudaSuccess) return e;
    if (wave == 0) return cudaErrorInvalidConfiguration;
    const uint32_t tiles = (a.rows + kTileRows - 1) / kTileRows;
    k<<<tiles < wave ? tiles : (uint32_t)wave, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <bool CF8>
cudaError_t launch_dynamic(const GatherArgs& a, float* scales, cudaStream_t stream) {
    constexpr auto k = gather_dynamic_kernel<CF8>;
    const size_t smem = sizeof(uint32_t) * ((size_t)a.B + 1);
    uint64_t wave = 0;
    const cudaError_t e = wave_ctas<k>(kThreads, smem, wave);
    if (e != cudaSuccess) return e;
    if (wave == 0) return cudaErrorInvalidConfiguration;
    const uint32_t ctas = (a.rows + kDynRows * (kThreads / 32) - 1) / (kDynRows * (kThreads / 32));
    k<<<ctas < wave ? ctas : (uint32_t)wave, kThreads, smem, stream>>>(a, scales);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host checks shared by both entry points; fills `a` (out left null).
int make_args(const kvw_paged_cache_t* cache, uint32_t layer_idx, const uint32_t* ctx_offsets,
              uint32_t num_batches, uint32_t total_rows, uint32_t* err_flags, GatherArgs& a) {
    if (cache->dtype != KVW_DTYPE_BF16 && cache->dtype != KVW_DTYPE_FP8_E4M3) return KVW_EUNSUPPORTED;
    if (cache->head_size != kRow || cache->num_heads != 1) return KVW_EUNSUPPORTED;
    if (num_batches > KVW_MAX_BATCHES) return KVW_EUNSUPPORTED;
    const bool cf8 = cache->dtype == KVW_DTYPE_FP8_E4M3;
    const int64_t esz = cf8 ? 1 : 2;
    if (!ctx_offsets || !cache->data || !cache->page_table) return KVW_EINVAL;
    if (layer_idx >= cache->num_layers || cache->page_size == 0 || cache->max_pages_per_seq == 0)
        return KVW_EINVAL;
    if (cf8 && !(cache->scale > 0.0f && cache->scale < 3.0e38f)) return KVW_EINVAL;
    if (!aligned16(cache->data)) return KVW_EINVAL;
    if ((cache->stride_page * esz) % 16 || (cache->stride_layer * esz) % 16 ||
        (cache->stride_token * esz) % 16 || cache->stride_page <= 0 || cache->stride_token <= 0)
        return KVW_EINVAL;
    a.out = nullptr;
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
    a.ps_div = make_fast_div(cache->page_size);
    a.cache_scale = cache->scale;
    a.out_scale = 1.0f;
    return KVW_OK;
}

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
    GatherArgs a;
    const int st = make_args(cache, layer_idx, ctx_offsets, num_batches, total_rows, err_flags, a);
    if (st != KVW_OK) return st;
    if (total_rows == 0) return KVW_OK;
    const bool cf8 = cache->dtype == KVW_DTYPE_FP8_E4M3, of8 = out_dtype == KVW_DTYPE_FP8_E4M3;
    if (!out || !aligned16(out)) return KVW_EINVAL;
    if (of8 && !(out_scale > 0.0f && out_scale < 3.0e38f)) return KVW_EINVAL;
    a.out = static_cast<unsigned char*>(out);
    a.out_scale = out_scale;
    const cudaError_t e = cf8 ? (of8 ? launch<true, true>(a, stream) : launch<true, false>(a, stream))
                              : (of8 ? launch<false, true>(a, stream) : launch<false, false>(a, stream));
    return e == cudaSuccess ? KVW_OK : KVW_ECUDA;
}

extern "C" int kvw_mla_gather_latent_fp8_dynamic(void* out_codes, float* out_scales,
                                                 const kvw_paged_cache_t* cache,
                                                 uint32_t layer_idx, const uint32_t* ctx_offsets,
                                                 uint32_t num_batches, uint32_t total_rows,
                                                 uint32_t* err_flags, cudaStream_t stream) {
    using namespace kvw;
    if (!cache) return KVW_EINVAL;
    GatherArgs a;
    const int st = make_args(cache, layer_idx, ctx_offsets, num_batches, total_rows, err_flags, a);
    if (st != KVW_OK) return st;
    if (total_rows == 0) return KVW_OK;
    if (!out_codes || !out_scales || !aligned16(out_codes) ||
        (reinterpret_cast<uintptr_t>(out_scales) & 3u) != 0)
        return KVW_EINVAL;
    a.out = static_cast<unsigned char*>(out_codes);
    const cudaError_t e = cache->dtype == KVW_DTYPE_FP8_E4M3
                              ? launch_dynamic<true>(a, out_scales, stream)
                              : launch_dynamic<false>(a, out_scales, stream);
    return e == cudaSuccess ? KVW_OK : KVW_ECUDA;
}
