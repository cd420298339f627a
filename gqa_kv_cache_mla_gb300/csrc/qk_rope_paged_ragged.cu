// Fused GQA Q/K RoPE: rotate every query head of the new tokens into
// `output` and every key head of their cache slots in place.
//
// Operation: "generic_fused_qk_rope_bshd_paged_ragged" (Modular MAX kernel
// API, Mojo function page: description (Q rotated into output, K rotated in
// the paged K cache after the fused QKV projection); Parameters interleaved,
// has_position_ids, mrope_section; Args q_proj, input_row_offsets,
// kv_collection, freqs_cis, position_ids, layer_idx, output).
//
// GB300 design.  A token is (Hq + Hk) heads x head_size/16 "items"; an item
// is 8 rotary pairs = two 16-byte vectors (adjacent for interleaved pairs,
// k and k + head_size/2 for half-split pairs).  The CTA has one thread per
// item of a token (rounded up to whole warps), so a thread's head and pair
// range never change, and it walks TPB consecutive tokens:
//   phase 0  query threads issue all their q_proj loads (TPB x 32 B);
//   phase 1  offsets/cache_lengths staged and validated in shared memory;
//   phase 2  per token: slot position and page lookup, and the token's
//            composed freqs row (pair k read from the row of its own
//            position, which covers plain, position_ids and mrope cases) is
//            gathered once into shared memory;
//   phase 3  key threads load their slot rows, everybody rotates and stores.
// Every rotation is done in fp32 with separately rounded products and the
// result is rounded once to bf16.
#include <cstdint>

#include "kvw_device.cuh"

namespace kvw {
namespace {

constexpr uint32_t kMaxHead = 512;

struct GqaArgs {
    const uint16_t* q_in;  // bf16 [T, Hq, S]
    uint16_t* q_out;       // bf16 [T, Hq, S], may alias q_in
    uint16_t* cache;       // bf16
    const uint32_t* offsets;
    const uint32_t* cache_lengths;
    const uint32_t* page_table;
    const uint32_t* position_ids;  // [T] or [3, T] or null
    const float* freqs;            // [freqs_rows, S]
    uint32_t* err_flags;
    int64_t s_page, s_token, s_head, layer_off;
    uint32_t B, T, Hq, Hk, S, freqs_rows, max_pages, num_pages, page_size;
    uint32_t mode;         // 0: slot positions, 1: position_ids[T], 2: mrope [3, T]
    uint32_t sec0, sec01;  // mrope section ends, in pairs
    uint32_t items;        // (Hq + Hk) * S / 16
};

__device__ __forceinline__ uint32_t section_of(const GqaArgs& a, uint32_t k) {
    return k < a.sec0 ? 0u : (k < a.sec01 ? 1u : 2u);
}

template <bool INTERLEAVED, int TPB>
__global__ void __launch_bounds__(1024) qk_rope_kernel(const GqaArgs a) {
    extern __shared__ uint32_t s_dyn[];
    uint32_t* s_off = s_dyn;
    uint32_t* s_clen = s_dyn + a.B + 1;
    __shared__ __align__(16) float s_cs[TPB][kMaxHead];  // composed (cos, sin) per pair
    __shared__ int64_t s_kbase[TPB];
    __shared__ int s_bad[TPB];

    const uint32_t groups = a.S >> 4;  // items per head
    const uint32_t i = threadIdx.x;
    const bool has_item = i < a.items;
    const uint32_t h = has_item ? i / groups : 0u;
    const uint32_t m = has_item ? i % groups : 0u;
    const bool is_q = has_item && h < a.Hq;
    const uint32_t t_begin = blockIdx.x * TPB;
    // element offsets of the two vectors of this item inside a head row
    const uint32_t e0 = INTERLEAVED ? 16u * m : 8u * m;
    const uint32_t e1 = INTERLEAVED ? 16u * m + 8u : (a.S >> 1) + 8u * m;

    if (i < TPB) s_bad[i] = 0;

    // phase 0: query data
    uint4 xa[TPB], xb[TPB];
#pragma unroll
    for (int u = 0; u < TPB; ++u) {
        xa[u] = make_uint4(0, 0, 0, 0);
        xb[u] = xa[u];
        const uint32_t t = t_begin + u;
        if (is_q && t < a.T) {
            const uint16_t* row = a.q_in + ((uint64_t)t * a.Hq + h) * a.S;
            xa[u] = ld_stream(reinterpret_cast<const uint4*>(row + e0));
            xb[u] = ld_stream(reinterpret_cast<const uint4*>(row + e1));
        }
    }

    // phase 1: ragged metadata (contains a __syncthreads, so s_bad is ready)
    if (!stage_ragged(a.offsets, a.cache_lengths, a.B, a.T, s_off, s_clen)) {
        if (threadIdx.x == 0) flag(a.err_flags, KVW_ERR_OFFSETS);
        return;
    }

    // phase 2a: slot row of each token
    if (i < TPB) {
        const uint32_t t = t_begin + i;
        int64_t base = -1;
        if (t < a.T) {
            const uint32_t b = find_request(s_off, a.B, t);
            const uint64_t pos = (uint64_t)s_clen[b] + (t - s_off[b]);
            base = slot_row(a.page_table, a.max_pages, a.num_pages, a.page_size, a.s_page,
                            a.s_token, a.layer_off, b, pos);
        }
        s_kbase[i] = base;
    }
    // phase 2b: composed freqs rows, one (cos, sin) pair per rotary pair
    const uint32_t half = a.S >> 1;
    for (uint32_t idx = threadIdx.x; idx < TPB * half; idx += blockDim.x) {
        const uint32_t u = idx / half, k = idx % half;
        const uint32_t t = t_begin + u;
        if (t >= a.T) continue;
        uint64_t p;
        if (a.mode == 0) {
            const uint32_t b = find_request(s_off, a.B, t);
            p = (uint64_t)s_clen[b] + (t - s_off[b]);
        } else if (a.mode == 1) {
            p = __ldg(a.position_ids + t);
        } else {
            p = __ldg(a.position_ids + (uint64_t)section_of(a, k) * a.T + t);
        }
        float2 cs = make_float2(0.f, 0.f);
        if (p < a.freqs_rows)
            cs = __ldg(reinterpret_cast<const float2*>(a.freqs + p * a.S) + k);
        else
            s_bad[u] = 1;
        *reinterpret_cast<float2*>(&s_cs[u][2 * k]) = cs;
    }
    __syncthreads();

    // phase 3a: key data (needs the slot rows)
    if (has_item && !is_q) {
#pragma unroll
        for (int u = 0; u < TPB; ++u) {
            const int64_t kb = s_kbase[u];
            if (kb >= 0 && !s_bad[u]) {
                const uint16_t* row = a.cache + kb + (int64_t)(h - a.Hq) * a.s_head;
                xa[u] = *reinterpret_cast<const uint4*>(row + e0);
                xb[u] = *reinterpret_cast<const uint4*>(row + e1);
            }
        }
    }
    if (i < TPB && t_begin + i < a.T) {
        if (s_bad[i])
            flag(a.err_flags, KVW_ERR_POSITION);
        else if (s_kbase[i] < 0)
            flag(a.err_flags, KVW_ERR_PAGE);
    }
    if (!has_item) return;

    // phase 3b: rotate and store
#pragma unroll
    for (int u = 0; u < TPB; ++u) {
        const uint32_t t = t_begin + u;
        if (t >= a.T || s_bad[u]) continue;
        if (!is_q && s_kbase[u] < 0) continue;
        const float4* cs4 = reinterpret_cast<const float4*>(&s_cs[u][16u * m]);
        const float4 c0 = cs4[0], c1 = cs4[1], c2 = cs4[2], c3 = cs4[3];
        const float c[8] = {c0.x, c0.z, c1.x, c1.z, c2.x, c2.z, c3.x, c3.z};
        const float s[8] = {c0.y, c0.w, c1.y, c1.w, c2.y, c2.w, c3.y, c3.w};
        float va[8], vb[8], ya[8], yb[8];
        unpack8(xa[u], va);
        unpack8(xb[u], vb);
        if (INTERLEAVED) {  // pairs (va0,va1) (va2,va3) .. (vb6,vb7)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                rope_pair(va[2 * q], va[2 * q + 1], c[q], s[q], ya[2 * q], ya[2 * q + 1]);
                rope_pair(vb[2 * q], vb[2 * q + 1], c[q + 4], s[q + 4], yb[2 * q], yb[2 * q + 1]);
            }
        } else {  // pairs (va[q], vb[q])
#pragma unroll
            for (int q = 0; q < 8; ++q) rope_pair(va[q], vb[q], c[q], s[q], ya[q], yb[q]);
        }
        uint16_t* row = is_q ? a.q_out + ((uint64_t)t * a.Hq + h) * a.S
                             : a.cache + s_kbase[u] + (int64_t)(h - a.Hq) * a.s_head;
        if (is_q) {
            st_stream(reinterpret_cast<uint4*>(row + e0), pack8_bf16(ya));
            st_stream(reinterpret_cast<uint4*>(row + e1), pack8_bf16(yb));
        } else {
            *reinterpret_cast<uint4*>(row + e0) = pack8_bf16(ya);
            *reinterpret_cast<uint4*>(row + e1) = pack8_bf16(yb);
        }
    }
}

template <bool INTERLEAVED, int TPB>
cudaError_t launch(const GqaArgs& a, uint32_t threads, size_t smem, cudaStream_t stream) {
    auto k = qk_rope_kernel<INTERLEAVED, TPB>;
    if (smem > 16 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const uint32_t blocks = (a.T + TPB - 1) / TPB;
    k<<<blocks, threads, smem, stream>>>(a);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvw

extern "C" int kvw_qk_rope_paged_ragged(const void* q_proj, const uint32_t* input_row_offsets,
                                        uint32_t num_batches, uint32_t tot_seq_len,
                                        uint32_t num_q_heads, const kvw_paged_cache_t* cache,
                                        const void* freqs_cis, uint32_t freqs_rows,
                                        const uint32_t* position_ids, int interleaved,
                                        const uint32_t* mrope_section, uint32_t layer_idx,
                                        void* output, uint32_t* err_flags, cudaStream_t stream) {
    using namespace kvw;
    if (!cache) return KVW_EINVAL;
    if (cache->dtype != KVW_DTYPE_BF16) return KVW_EUNSUPPORTED;
    const uint32_t S = cache->head_size;
    if (S == 0 || S % 16 != 0 || S > kMaxHead) return KVW_EUNSUPPORTED;
    if (num_batches > KVW_MAX_BATCHES) return KVW_EUNSUPPORTED;
    const uint64_t items = (uint64_t)(num_q_heads + (uint64_t)cache->num_heads) * (S / 16);
    if (items > 1024) return KVW_EUNSUPPORTED;
    uint32_t sec0 = 0, sec01 = 0;
    if (mrope_section) {
        if (!position_ids) return KVW_EINVAL;
        const uint64_t sum = (uint64_t)mrope_section[0] + mrope_section[1] + mrope_section[2];
        if (sum != S / 2) return KVW_EINVAL;
        sec0 = mrope_section[0];
        sec01 = mrope_section[0] + mrope_section[1];
    }
    if (tot_seq_len == 0) return KVW_OK;
    if (!input_row_offsets || !freqs_cis || !cache->data || !cache->page_table ||
        !cache->cache_lengths)
        return KVW_EINVAL;
    if (num_q_heads > 0 && (!q_proj || !output)) return KVW_EINVAL;
    if (layer_idx >= cache->num_layers || cache->page_size == 0 || freqs_rows == 0 ||
        cache->max_pages_per_seq == 0)
        return KVW_EINVAL;
    if (!aligned16(freqs_cis) || !aligned16(cache->data) ||
        (num_q_heads > 0 && (!aligned16(q_proj) || !aligned16(output))))
        return KVW_EINVAL;
    if ((cache->stride_page * 2) % 16 || (cache->stride_layer * 2) % 16 ||
        (cache->stride_token * 2) % 16 || (cache->stride_head * 2) % 16 ||
        cache->stride_page <= 0 || cache->stride_token <= 0)
        return KVW_EINVAL;
    if (items == 0) return KVW_OK;

    GqaArgs a;
    a.q_in = static_cast<const uint16_t*>(q_proj);
    a.q_out = static_cast<uint16_t*>(output);
    a.cache = static_cast<uint16_t*>(cache->data);
    a.offsets = input_row_offsets;
    a.cache_lengths = cache->cache_lengths;
    a.page_table = cache->page_table;
    a.position_ids = position_ids;
    a.freqs = static_cast<const float*>(freqs_cis);
    a.err_flags = err_flags;
    a.s_page = cache->stride_page;
    a.s_token = cache->stride_token;
    a.s_head = cache->stride_head;
    a.layer_off = (int64_t)layer_idx * cache->stride_layer;
    a.B = num_batches;
    a.T = tot_seq_len;
    a.Hq = num_q_heads;
    a.Hk = cache->num_heads;
    a.S = S;
    a.freqs_rows = freqs_rows;
    a.max_pages = cache->max_pages_per_seq;
    a.num_pages = cache->num_pages;
    a.page_size = cache->page_size;
    a.mode = position_ids ? (mrope_section ? 2u : 1u) : 0u;
    a.sec0 = sec0;
    a.sec01 = sec01;
    a.items = (uint32_t)items;

    const uint32_t threads = (uint32_t)((items + 31) / 32 * 32);
    const size_t smem = sizeof(uint32_t) * (2 * (size_t)num_batches + 1);
    // Tokens per CTA: enough to keep >= 2 waves of CTAs over 152 SMs.
    int tpb = 4;
    while (tpb > 1 && (uint64_t)(tot_seq_len + tpb - 1) / tpb < 152ull * 4) tpb >>= 1;
    cudaError_t e;
    if (interleaved) {
        e = tpb == 4 ? launch<true, 4>(a, threads, smem, stream)
          : tpb == 2 ? launch<true, 2>(a, threads, smem, stream)
                     : launch<true, 1>(a, threads, smem, stream);
    } else {
        e = tpb == 4 ? launch<false, 4>(a, threads, smem, stream)
          : tpb == 2 ? launch<false, 2>(a, threads, smem, stream)
                     : launch<false, 1>(a, threads, smem, stream);
    }
    return e == cudaSuccess ? KVW_OK : KVW_ECUDA;
}
