// Fused MLA key-cache write: RoPE on q_rope and on the rope part of each
// latent row, RMSNorm of the 512-wide latent part, quantisation to the cache
// type and scatter through the page table.
//
// Operation: "mla_fused_rope_rmsnorm_quantization" (Modular MAX kernel API,
// Mojo function page: description of the three fused operations; Args
// q_rope_output, q_rope, input_row_offsets, freqs_cis, gamma, kv_collection,
// layer_idx, epsilon; Parameters kv_input_fn) and the
// fused_rope_rmsnorm_quantization_kernel entry of the "mla_graph" module page.
//
// GB300 design.  The launch is purely HBM-bound (about 0.5 flop per byte),
// so the kernel is organised around keeping enough 16-byte loads in flight on
// all SMs:
//   * CTAs [0, kv_blocks) own latent rows, one warp per token: lane l holds
//     columns 8l..8l+7 and 256+8l..256+8l+7 of the latent part (lanes 0..7
//     also one 8-wide slice of the rope part), a 5-step xor-shuffle gives the
//     sum of squares, and the row leaves as one coalesced 576 B (FP8) or
//     1152 B (bf16) store into its page slot.
//   * the remaining CTAs stream q_rope as a flat array of 16-byte vectors,
//     VPT vectors per thread, all loads issued before the ragged lookup so
//     the lookup's latency hides under them.  A head row is 8 vectors and
//     256 % 8 == 0, so a thread always works on the same 8 columns and needs
//     one freqs slice per token.
//   * every CTA stages input_row_offsets and cache_lengths in shared memory,
//     validates them and binary-searches its tokens' requests there.
// Both roles live in one launch so a decode step is one kernel.
// Decode fast path: when the batch has as many tokens as requests, the
// offsets are most likely the identity (one new token per request), so
// token t is request t at slot position cache_lengths[t].  A CTA then loads
// cache_lengths first, issues the dependent page-table and freqs loads
// straight from registers (no staging, search or barrier in between), and
// checks the identity over the whole offsets table with one block vote taken
// while those loads are in flight; a CTA that finds anything else runs the
// general path above, so results and flags are the same either way.
#include <cstdint>

#include "kvw_device.cuh"

namespace kvw {
namespace {

constexpr uint32_t kThreads = 256;
constexpr uint32_t kRowsPerKvBlock = kThreads / 32;  // one warp per latent row
constexpr uint32_t kNorm = 512, kRope = 64, kRow = kNorm + kRope;

struct MlaArgs {
    const uint4* q_in;   // bf16 [T, H, 64] as 16-byte vectors
    uint4* q_out;        // bf16 [T, H, 64]
    const uint16_t* kv_in;
    int64_t kv_row_stride;  // elements
    const uint32_t* offsets;
    const uint32_t* cache_lengths;
    const uint32_t* page_table;
    const float* freqs;  // [freqs_rows, 64]
    const uint4* gamma;  // bf16 [512]
    void* cache;
    uint32_t* err_flags;
    int64_t s_page, s_token, layer_off;  // elements of the cache type
    uint32_t q_vectors;                  // T * H * 8
    uint32_t B, T, H, freqs_rows, max_pages, num_pages, page_size;
    uint32_t kv_blocks;
    uint32_t decode;  // T == B: try the one-token-per-request fast path first
    float eps, scale;
    FastDiv ps_div;   // division by page_size
    FastDiv vpt_div;  // division by the 16-byte q vectors per token (H * 8)
};

// Stage offsets[0..B] and cache_lengths[0..B-1] in shared memory and check
// that the offsets start at 0, never decrease and end at T (uniform verdict).
// Copy, barrier, check from shared memory, barrier: for the many short CTAs
// of a prefill launch this form measured faster than checking from
// registers before a single barrier.
__device__ __forceinline__ bool stage_tables(const uint32_t* __restrict__ offsets,
                                             const uint32_t* __restrict__ cache_lengths,
                                             uint32_t B, uint32_t T, uint32_t* s_off,
                                             uint32_t* s_clen) {
    for (uint32_t i = threadIdx.x; i <= B; i += blockDim.x) {
        s_off[i] = __ldg(offsets + i);
        if (i < B) s_clen[i] = __ldg(cache_lengths + i);
    }
    __syncthreads();
    int ok = 1;
    for (uint32_t i = threadIdx.x; i < B; i += blockDim.x)
        if (s_off[i] > s_off[i + 1]) ok = 0;
    if (threadIdx.x == 0 && (s_off[0] != 0u || s_off[B] != T)) ok = 0;
    return __syncthreads_and(ok) != 0;
}

template <bool FP8>
__device__ __forceinline__ void store8(void* cache, int64_t elem, const float (&y)[8], float scale) {
    if constexpr (FP8) {
        float z[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) z[i] = scale == 1.0f ? y[i] : __fdiv_rn(y[i], scale);
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + elem) = pack8_e4m3(z);
    } else {
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(cache) + elem) = pack8_bf16(y);
    }
}

// The row work of one warp once its slot is known: RMSNorm of the 512 latent
// values (16 per lane), RoPE of the rope part (lanes 0..7, 4 adjacent pairs
// each, freqs slice in fa/fb), quantisation and the store of the 576-wide
// cache row at element offset `base`.  x0/x1/xr hold the input row (unused
// when INPLACE: the row is read from its slot), g0/g1 this lane's gamma.
template <bool FP8, bool INPLACE>
__device__ __forceinline__ void latent_row_compute(const MlaArgs& a, int64_t base, uint32_t lane,
                                                   const uint4& x0, const uint4& x1,
                                                   const uint4& xr, const uint4& g0,
                                                   const uint4& g1, const float4& fa,
                                                   const float4& fb) {
    float v0[8], v1[8], w0[8], w1[8], xv[8];
    if (INPLACE) {
        constexpr int64_t esz = FP8 ? 1 : 2;
        const unsigned char* rowb = static_cast<const unsigned char*>(a.cache) + base * esz;
        load_k8<FP8>(rowb + (int64_t)lane * 8 * esz, v0, a.scale);
        load_k8<FP8>(rowb + (int64_t)(256 + lane * 8) * esz, v1, a.scale);
        if (lane < 8) load_k8<FP8>(rowb + (int64_t)(kNorm + lane * 8) * esz, xv, a.scale);
    } else {
        unpack8(x0, v0);
        unpack8(x1, v1);
        unpack8(xr, xv);
    }
    unpack8(g0, w0);
    unpack8(g1, w1);
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(v0[i], v0[i]));
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(v1[i], v1[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float r = rms_inv(ss, (float)kNorm, a.eps);
    float y0[8], y1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        y0[i] = __fmul_rn(__fmul_rn(v0[i], r), w0[i]);
        y1[i] = __fmul_rn(__fmul_rn(v1[i], r), w1[i]);
    }
    store8<FP8>(a.cache, base + lane * 8, y0, a.scale);
    store8<FP8>(a.cache, base + 256 + lane * 8, y1, a.scale);
    if (lane < 8) {  // rope part: 4 adjacent pairs per lane
        float yr[8];
        rope_pair(xv[0], xv[1], fa.x, fa.y, yr[0], yr[1]);
        rope_pair(xv[2], xv[3], fa.z, fa.w, yr[2], yr[3]);
        rope_pair(xv[4], xv[5], fb.x, fb.y, yr[4], yr[5]);
        rope_pair(xv[6], xv[7], fb.z, fb.w, yr[6], yr[7]);
        store8<FP8>(a.cache, base + kNorm + lane * 8, yr, a.scale);
    }
}

// Input row (not INPLACE) and gamma slices of this lane.
template <bool INPLACE>
__device__ __forceinline__ void latent_row_loads(const MlaArgs& a, uint32_t t, uint32_t lane,
                                                 uint4& x0, uint4& x1, uint4& xr, uint4& g0,
                                                 uint4& g1) {
    if (!INPLACE) {
        const uint4* row = reinterpret_cast<const uint4*>(a.kv_in + (int64_t)t * a.kv_row_stride);
        x0 = ld_stream(row + lane);
        x1 = ld_stream(row + 32 + lane);
        if (lane < 8) xr = ld_stream(row + 64 + lane);
    }
    g0 = ld_table(a.gamma + lane);
    g1 = ld_table(a.gamma + 32 + lane);
}

// One warp per token: RMSNorm of the latent part, RoPE of the rope part,
// quantise, write the 576-wide cache row.
// INPLACE: the latent row is not read from kv_in but from the cache slot
// it is written back to (bf16, or E4M3 dequantised with the cache scale).
template <bool FP8, bool INPLACE>
__device__ __forceinline__ void latent_rows(const MlaArgs& a, uint32_t* s_off, uint32_t* s_clen) {
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t t = blockIdx.x * kRowsPerKvBlock + warp;
    const bool active = t < a.T;
    uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0, xr = x0, g0 = x0, g1 = x0;
    if (active) latent_row_loads<INPLACE>(a, t, lane, x0, x1, xr, g0, g1);
    if (!stage_tables(a.offsets, a.cache_lengths, a.B, a.T, s_off, s_clen)) {
        if (threadIdx.x == 0) flag(a.err_flags, KVW_ERR_OFFSETS);
        return;
    }
    if (!active) return;
    const uint32_t b = find_request(s_off, a.B, t);
    const uint64_t pos = (uint64_t)s_clen[b] + (t - s_off[b]);
    if (pos >= a.freqs_rows) {
        if (lane == 0) flag(a.err_flags, KVW_ERR_POSITION);
        return;
    }
    const int64_t base = slot_row(a.page_table, a.max_pages, a.num_pages, a.ps_div, a.s_page,
                                  a.s_token, a.layer_off, b, pos);
    if (base < 0) {
        if (lane == 0) flag(a.err_flags, KVW_ERR_PAGE);
        return;
    }
    float4 fa = make_float4(0.f, 0.f, 0.f, 0.f), fb = fa;
    if (lane < 8) {
        const float4* fr = reinterpret_cast<const float4*>(a.freqs + pos * kRope) + lane * 2;
        fa = ld_table(fr);
        fb = ld_table(fr + 1);
    }
    latent_row_compute<FP8, INPLACE>(a, base, lane, x0, x1, xr, g0, g1, fa, fb);
}

// Whether input_row_offsets[i] == i for the entries this thread checks
// (i = threadIdx.x, + blockDim.x, ... <= B); the loads are issued here and
// the vote is taken later.
__device__ __forceinline__ uint32_t identity_part(const uint32_t* __restrict__ offsets,
                                                  uint32_t B) {
    uint32_t ok = 1;
    for (uint32_t i = threadIdx.x; i <= B; i += kThreads) ok &= __ldg(offsets + i) == i ? 1u : 0u;
    return ok;
}

// Decode fast path of the latent CTAs (T == B).  Returns false, before
// writing or flagging anything, when the offsets are not the identity; the
// CTA then runs latent_rows.  Uniform across the CTA.
template <bool FP8, bool INPLACE>
__device__ __forceinline__ bool latent_rows_decode(const MlaArgs& a) {
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t t = blockIdx.x * kRowsPerKvBlock + warp;
    const bool active = t < a.T;
    const uint32_t ok = identity_part(a.offsets, a.B);
    const uint32_t pos = active ? __ldg(a.cache_lengths + t) : 0u;
    uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0, xr = x0, g0 = x0, g1 = x0;
    if (active) latent_row_loads<INPLACE>(a, t, lane, x0, x1, xr, g0, g1);
    const bool pos_ok = pos < a.freqs_rows;
    const uint32_t pidx = fast_div(pos, a.ps_div);
    uint32_t page = KVW_PAGE_UNMAPPED;
    float4 fa = make_float4(0.f, 0.f, 0.f, 0.f), fb = fa;
    if (active && pos_ok) {
        if (pidx < a.max_pages) page = __ldg(a.page_table + (uint64_t)t * a.max_pages + pidx);
        if (lane < 8) {
            const float4* fr =
                reinterpret_cast<const float4*>(a.freqs + (uint64_t)pos * kRope) + lane * 2;
            fa = ld_table(fr);
            fb = ld_table(fr + 1);
        }
    }
    if (!__syncthreads_and(ok)) return false;
    if (!active) return true;
    if (!pos_ok) {
        if (lane == 0) flag(a.err_flags, KVW_ERR_POSITION);
        return true;
    }
    if (page >= a.num_pages) {
        if (lane == 0) flag(a.err_flags, KVW_ERR_PAGE);
        return true;
    }
    const int64_t base =
        (int64_t)page * a.s_page + a.layer_off + (int64_t)(pos - pidx * a.page_size) * a.s_token;
    latent_row_compute<FP8, INPLACE>(a, base, lane, x0, x1, xr, g0, g1, fa, fb);
    return true;
}

// Rotation of one q_rope vector (8 columns, 4 adjacent pairs) and its store.
template <bool QF8>
__device__ __forceinline__ void q_vector_compute(const MlaArgs& a, uint32_t v, const uint4& x,
                                                 const float4& fa, const float4& fb) {
    float xv[8], y[8];
    unpack8(x, xv);
    rope_pair(xv[0], xv[1], fa.x, fa.y, y[0], y[1]);
    rope_pair(xv[2], xv[3], fa.z, fa.w, y[2], y[3]);
    rope_pair(xv[4], xv[5], fb.x, fb.y, y[4], y[5]);
    rope_pair(xv[6], xv[7], fb.z, fb.w, y[6], y[7]);
    if (QF8)
        reinterpret_cast<uint2*>(a.q_out)[v] = pack8_e4m3(y);
    else
        st_stream(a.q_out + v, pack8_bf16(y));
}

// Decode fast path of the q CTAs (T == B), same contract as
// latent_rows_decode.  Every token's first vector reports a bad position,
// so the flag is raised once per token, as in q_rows.
template <int VPT, bool QF8>
__device__ __forceinline__ bool q_rows_decode(const MlaArgs& a) {
    const uint32_t qb = blockIdx.x - a.kv_blocks;
    const uint32_t vbase = qb * (kThreads * VPT);
    const uint32_t vpt = a.H * 8u;  // vectors per token
    const uint32_t ok = identity_part(a.offsets, a.B);
    uint32_t pos[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const uint32_t v = vbase + threadIdx.x + i * kThreads;
        pos[i] = v < a.q_vectors ? __ldg(a.cache_lengths + fast_div(v, a.vpt_div)) : 0xffffffffu;
    }
    uint4 x[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const uint32_t v = vbase + threadIdx.x + i * kThreads;
        x[i] = v < a.q_vectors ? ld_stream(a.q_in + v) : make_uint4(0, 0, 0, 0);
    }
    const uint32_t j = threadIdx.x & 7u;  // 8-column slice of the 64-wide head row
    float4 fa[VPT], fb[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        fa[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        fb[i] = fa[i];
        if (pos[i] < a.freqs_rows) {
            const float4* fr =
                reinterpret_cast<const float4*>(a.freqs + (uint64_t)pos[i] * kRope) + j * 2;
            fa[i] = ld_table(fr);
            fb[i] = ld_table(fr + 1);
        }
    }
    if (!__syncthreads_and(ok)) return false;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const uint32_t v = vbase + threadIdx.x + i * kThreads;
        if (v >= a.q_vectors) break;
        if (pos[i] >= a.freqs_rows) {
            if (v % vpt == 0u) flag(a.err_flags, KVW_ERR_POSITION);
            continue;
        }
        q_vector_compute<QF8>(a, v, x[i], fa[i], fb[i]);
    }
    return true;
}

// q_rope streaming: VPT 16-byte vectors per thread.
// QF8: q_rope_output is E4M3 (direct saturating conversion) instead of bf16.
template <int VPT, bool QF8>
__device__ __forceinline__ void q_rows(const MlaArgs& a, uint32_t* s_off, uint32_t* s_clen) {
    __shared__ uint32_t s_pos[(kThreads * VPT) / 8 + 2];
    const uint32_t qb = blockIdx.x - a.kv_blocks;
    const uint32_t vbase = qb * (kThreads * VPT);
    uint4 x[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) x[i] = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const uint32_t v = vbase + threadIdx.x + i * kThreads;
        if (v < a.q_vectors) x[i] = ld_stream(a.q_in + v);
    }
    if (!stage_tables(a.offsets, a.cache_lengths, a.B, a.T, s_off, s_clen)) {
        if (threadIdx.x == 0) flag(a.err_flags, KVW_ERR_OFFSETS);
        return;
    }
    const uint32_t vpt = a.H * 8u;  // vectors per token
    const uint32_t t0 = fast_div(vbase, a.vpt_div);
    const uint32_t vlast = min(vbase + kThreads * VPT, a.q_vectors) - 1u;
    const uint32_t ntok = fast_div(vlast, a.vpt_div) - t0 + 1u;
    for (uint32_t k = threadIdx.x; k < ntok; k += kThreads) {
        const uint32_t t = t0 + k;
        const uint32_t b = find_request(s_off, a.B, t);
        const uint64_t pos = (uint64_t)s_clen[b] + (t - s_off[b]);
        if (pos >= a.freqs_rows) {
            s_pos[k] = 0xffffffffu;
            flag(a.err_flags, KVW_ERR_POSITION);
        } else {
            s_pos[k] = (uint32_t)pos;
        }
    }
    __syncthreads();
    const uint32_t j = threadIdx.x & 7u;  // 8-column slice of the 64-wide head row
    uint32_t cur_t = 0xffffffffu, p = 0xffffffffu;
    float4 fa = make_float4(0.f, 0.f, 0.f, 0.f), fb = fa;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const uint32_t v = vbase + threadIdx.x + i * kThreads;
        if (v >= a.q_vectors) break;
        const uint32_t t = fast_div(v, a.vpt_div);
        if (t != cur_t) {
            cur_t = t;
            p = s_pos[t - t0];
            if (p != 0xffffffffu) {
                const float4* fr = reinterpret_cast<const float4*>(a.freqs + (uint64_t)p * kRope) + j * 2;
                fa = ld_table(fr);
                fb = ld_table(fr + 1);
            }
        }
        if (p == 0xffffffffu) continue;
        q_vector_compute<QF8>(a, v, x[i], fa, fb);
    }
}

template <bool FP8, int VPT, bool QF8, bool INPLACE>
__global__ void __launch_bounds__(kThreads) mla_rope_rmsnorm_quant_kernel(const MlaArgs a) {
    extern __shared__ uint32_t s_dyn[];
    uint32_t* s_off = s_dyn;
    uint32_t* s_clen = s_dyn + a.B + 1;
    // the fast path exists in the one-wave instances (VPT 1 and 2) a decode
    // batch launches; the VPT 4 instances of long prefill launches keep their
    // register count without it
    constexpr bool kDecodePath = VPT <= 2;
    if (blockIdx.x < a.kv_blocks) {
        if (kDecodePath && a.decode && latent_rows_decode<FP8, INPLACE>(a)) return;
        latent_rows<FP8, INPLACE>(a, s_off, s_clen);
    } else {
        if (kDecodePath && a.decode && q_rows_decode<VPT, QF8>(a)) return;
        q_rows<VPT, QF8>(a, s_off, s_clen);
    }
}

template <bool FP8, int VPT, bool QF8, bool INPLACE>
cudaError_t launch(const MlaArgs& a, uint32_t blocks, size_t smem, cudaStream_t stream) {
    constexpr auto k = mla_rope_rmsnorm_quant_kernel<FP8, VPT, QF8, INPLACE>;
    const cudaError_t e = prepare_smem<k>(smem);
    if (e != cudaSuccess) return e;
    k<<<blocks, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

// CTAs of this kernel that fit on the device at once (all SMs).
template <bool FP8, int VPT, bool QF8, bool INPLACE>
uint64_t resident_ctas(size_t smem) {
    uint64_t n = 0;
    if (wave_ctas<mla_rope_rmsnorm_quant_kernel<FP8, VPT, QF8, INPLACE>>(kThreads, smem, n) !=
        cudaSuccess)
        return 0;
    return n;
}

// Grid sizing and launch of one instance.  Vectors per thread: the smallest
// of 1, 2, 4 whose grid fits in one wave of resident CTAs (a decode step is
// latency-bound: a second wave would double its duration); 4 when nothing
// fits (long prefill launches, where many short CTAs keep the memory system
// busy).
template <bool FP8, bool QF8, bool INPLACE>
cudaError_t launch_sized(const MlaArgs& a, uint64_t qvec, size_t smem, cudaStream_t stream) {
    int vpt = 4;
    for (int cand : {1, 2}) {
        const uint64_t qb = (qvec + (uint64_t)kThreads * cand - 1) / ((uint64_t)kThreads * cand);
        const uint64_t cap = cand == 1 ? resident_ctas<FP8, 1, QF8, INPLACE>(smem)
                                       : resident_ctas<FP8, 2, QF8, INPLACE>(smem);
        if (a.kv_blocks + qb <= cap) {
            vpt = cand;
            break;
        }
    }
    const uint64_t qblocks = (qvec + (uint64_t)kThreads * vpt - 1) / ((uint64_t)kThreads * vpt);
    const uint64_t blocks = a.kv_blocks + qblocks;
    if (blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
    return vpt == 1 ? launch<FP8, 1, QF8, INPLACE>(a, (uint32_t)blocks, smem, stream)
         : vpt == 2 ? launch<FP8, 2, QF8, INPLACE>(a, (uint32_t)blocks, smem, stream)
                    : launch<FP8, 4, QF8, INPLACE>(a, (uint32_t)blocks, smem, stream);
}

template <bool INPLACE>
cudaError_t dispatch(const MlaArgs& a, bool fp8, bool qf8, uint64_t qvec, size_t smem,
                     cudaStream_t stream) {
    if (fp8)
        return qf8 ? launch_sized<true, true, INPLACE>(a, qvec, smem, stream)
                   : launch_sized<true, false, INPLACE>(a, qvec, smem, stream);
    return qf8 ? launch_sized<false, true, INPLACE>(a, qvec, smem, stream)
               : launch_sized<false, false, INPLACE>(a, qvec, smem, stream);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvw

namespace kvw {
namespace {

// Validation and launch shared by the fused and the in-place entry points.
int mla_entry(void* q_rope_out, int32_t out_dtype, const void* q_rope,
              const uint32_t* input_row_offsets, uint32_t num_batches, uint32_t tot_seq_len,
              uint32_t num_heads, const void* freqs_cis, int32_t freq_dtype, uint32_t freqs_rows,
              const void* gamma, int32_t gamma_dtype, const void* kv_in, int64_t kv_row_stride,
              const kvw_paged_cache_t* cache, uint32_t layer_idx, float epsilon,
              uint32_t* err_flags, cudaStream_t stream, bool inplace) {
    if (!cache) return KVW_EINVAL;
    if ((out_dtype != KVW_DTYPE_BF16 && out_dtype != KVW_DTYPE_FP8_E4M3) ||
        freq_dtype != KVW_DTYPE_F32 || gamma_dtype != KVW_DTYPE_BF16)
        return KVW_EUNSUPPORTED;
    if (cache->dtype != KVW_DTYPE_BF16 && cache->dtype != KVW_DTYPE_FP8_E4M3) return KVW_EUNSUPPORTED;
    if (cache->head_size != kRow || cache->num_heads != 1) return KVW_EUNSUPPORTED;
    if (num_batches > KVW_MAX_BATCHES) return KVW_EUNSUPPORTED;
    if (tot_seq_len == 0) return KVW_OK;
    const bool fp8 = cache->dtype == KVW_DTYPE_FP8_E4M3;
    const bool qf8 = out_dtype == KVW_DTYPE_FP8_E4M3;
    const int64_t esz = fp8 ? 1 : 2;
    if (!input_row_offsets || !freqs_cis || !gamma || !cache->data || !cache->page_table ||
        !cache->cache_lengths)
        return KVW_EINVAL;
    if (!inplace && !kv_in) return KVW_EINVAL;
    if (num_heads > 0 && (!q_rope || !q_rope_out)) return KVW_EINVAL;
    if (layer_idx >= cache->num_layers || cache->page_size == 0 || freqs_rows == 0 ||
        cache->max_pages_per_seq == 0)
        return KVW_EINVAL;
    if (!(fp8 ? (cache->scale > 0.0f && cache->scale < 3.0e38f) : true) || !(epsilon >= 0.0f))
        return KVW_EINVAL;
    if (!inplace && (kv_row_stride < (int64_t)kRow || kv_row_stride % 8 != 0)) return KVW_EINVAL;
    if (!aligned16(freqs_cis) || !aligned16(gamma) || (!inplace && !aligned16(kv_in)) ||
        !aligned16(cache->data) ||
        (num_heads > 0 && (!aligned16(q_rope) || !aligned16(q_rope_out))))
        return KVW_EINVAL;
    if ((cache->stride_page * esz) % 16 || (cache->stride_layer * esz) % 16 ||
        (cache->stride_token * esz) % 16 || cache->stride_page <= 0 || cache->stride_token <= 0)
        return KVW_EINVAL;
    const uint64_t qvec = (uint64_t)tot_seq_len * num_heads * 8u;
    if (qvec > 0xfffff000ull) return KVW_EUNSUPPORTED;

    MlaArgs a;
    a.q_in = static_cast<const uint4*>(q_rope);
    a.q_out = static_cast<uint4*>(q_rope_out);
    a.kv_in = static_cast<const uint16_t*>(kv_in);
    a.kv_row_stride = kv_row_stride;
    a.offsets = input_row_offsets;
    a.cache_lengths = cache->cache_lengths;
    a.page_table = cache->page_table;
    a.freqs = static_cast<const float*>(freqs_cis);
    a.gamma = static_cast<const uint4*>(gamma);
    a.cache = cache->data;
    a.err_flags = err_flags;
    a.s_page = cache->stride_page;
    a.s_token = cache->stride_token;
    a.layer_off = (int64_t)layer_idx * cache->stride_layer;
    a.q_vectors = (uint32_t)qvec;
    a.B = num_batches;
    a.T = tot_seq_len;
    a.H = num_heads;
    a.freqs_rows = freqs_rows;
    a.max_pages = cache->max_pages_per_seq;
    a.num_pages = cache->num_pages;
    a.page_size = cache->page_size;
    a.kv_blocks = (tot_seq_len + kRowsPerKvBlock - 1) / kRowsPerKvBlock;
    a.decode = tot_seq_len == num_batches ? 1u : 0u;
    a.ps_div = make_fast_div(cache->page_size);
    a.vpt_div = make_fast_div(num_heads > 0 ? num_heads * 8u : 1u);
    a.eps = epsilon;
    a.scale = cache->scale;
    const size_t smem = sizeof(uint32_t) * (2 * (size_t)num_batches + 1);
    const cudaError_t e = inplace ? dispatch<true>(a, fp8, qf8, qvec, smem, stream)
                                  : dispatch<false>(a, fp8, qf8, qvec, smem, stream);
    return e == cudaSuccess ? KVW_OK : KVW_ECUDA;
}

}  // namespace
}  // namespace kvw

extern "C" int kvw_mla_rope_rmsnorm_quant(void* q_rope_out, int32_t out_dtype, const void* q_rope,
                                          const uint32_t* input_row_offsets, uint32_t num_batches,
                                          uint32_t tot_seq_len, uint32_t num_heads,
                                          const void* freqs_cis, int32_t freq_dtype,
                                          uint32_t freqs_rows, const void* gamma,
                                          int32_t gamma_dtype, const void* kv_in,
                                          int64_t kv_row_stride, const kvw_paged_cache_t* cache,
                                          uint32_t layer_idx, float epsilon, uint32_t* err_flags,
                                          cudaStream_t stream) {
    return kvw::mla_entry(q_rope_out, out_dtype, q_rope, input_row_offsets, num_batches,
                          tot_seq_len, num_heads, freqs_cis, freq_dtype, freqs_rows, gamma,
                          gamma_dtype, kv_in, kv_row_stride, cache, layer_idx, epsilon, err_flags,
                          stream, false);
}

extern "C" int kvw_mla_rope_rmsnorm_inplace(void* q_rope_out, int32_t out_dtype,
                                            const void* q_rope, const uint32_t* input_row_offsets,
                                            uint32_t num_batches, uint32_t tot_seq_len,
                                            uint32_t num_heads, const void* freqs_cis,
                                            int32_t freq_dtype, uint32_t freqs_rows,
                                            const void* gamma, int32_t gamma_dtype,
                                            const kvw_paged_cache_t* cache, uint32_t layer_idx,
                                            float epsilon, uint32_t* err_flags,
                                            cudaStream_t stream) {
    return kvw::mla_entry(q_rope_out, out_dtype, q_rope, input_row_offsets, num_batches,
                          tot_seq_len, num_heads, freqs_cis, freq_dtype, freqs_rows, gamma,
                          gamma_dtype, nullptr, 0, cache, layer_idx, epsilon, err_flags, stream,
                          true);
}
