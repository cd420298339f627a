// Fused GQA Q/K RoPE: rotate every query head of the new tokens into
// `output` and every key head of their cache slots in place.
//
// Operation: "generic_fused_qk_rope_bshd_paged_ragged" (Modular MAX kernel
// API, Mojo function page: description (Q rotated into output, K rotated in
// the paged K cache after the fused QKV projection); Parameters interleaved,
// has_position_ids, mrope_section; Args q_proj, input_row_offsets,
// kv_collection, freqs_cis, position_ids, layer_idx, output).
//
// GB300 design (slot positions and position_ids; mrope uses the
// register-staged kernel further down): a persistent, warp-specialised TMA
// pipeline.
//   * The tokens are cut into groups of TPB consecutive tokens; each CTA (one
//     per SM for a bf16 K cache, two for an E4M3 one, sized by shared memory)
//     walks groups blockIdx.x, + gridDim.x, ...
//   * A producer warp resolves each group's tokens (request by binary search
//     in the staged offsets, slot position, RoPE positions, page id) and
//     issues bulk (TMA) copies into a 2-stage shared-memory ring: the group's
//     q_proj rows (one copy, they are contiguous), the K rows (one copy per
//     run of adjacent slots) and the freqs_cis rows (one copy per run of
//     consecutive positions, or one per token with position_ids).
//     Copies complete on the stage's "full" mbarrier with a transaction
//     count, so no thread waits on individual loads.
//   * Twelve consumer warps (more measured no better, eight 2-4% slower) wait
//     for the stage, rotate from shared memory and
//     store straight to global memory (query rows to `output`, key rows back
//     to their slots), then release the stage on its "empty" mbarrier.  A
//     consumer thread owns one (token, 8-pair group, head slice): it reads the
//     group's 8 (cos, sin) pairs once and applies them to every head of its
//     slice.
// While the consumers work on one group, the copy engine is already filling
// the other stage, so every SM keeps tens of kilobytes in flight without
// holding them in registers.  Every wait is bounded (about one second) and
// reports KVW_ERR_TIMEOUT instead of hanging.
// Rotation arithmetic: fp32, separately rounded products, one rounding to
// bf16.
#include <cstdint>
#include <type_traits>

#include "kvw_device.cuh"

namespace kvw {
namespace {

constexpr uint32_t kMaxHead = 512;
constexpr int kConsumerWarps = 12;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStages = 2;
constexpr uint32_t kMaxTPB = 16;

struct GqaArgs {
    const uint16_t* q_in;  // bf16 [T, Hq, S]
    uint16_t* q_out;       // bf16 [T, Hq, S], may alias q_in
    unsigned char* cache;  // K/V cache bytes (bf16, or FP8 E4M3 with kscale)
    float kscale;          // FP8 dequantisation scale
    uint32_t kesz;         // bytes per cache element
    const uint32_t* offsets;
    const uint32_t* cache_lengths;
    const uint32_t* page_table;
    const uint32_t* position_ids;  // [T] or [3, T] or null
    const float* freqs;            // [freqs_rows, S]
    uint32_t* err_flags;
    int64_t s_page, s_token, s_head, layer_off;
    uint32_t B, T, Hq, Hk, S, freqs_rows, max_pages, num_pages, page_size;
    uint32_t mode;              // 0: slot positions, 1: position_ids[T], 2: mrope [3, T]
    uint32_t sec0, sec01;       // mrope section ends, in pairs
    uint32_t tpb, groups;       // tokens per group, number of groups
    uint32_t heads_contig;      // kv heads adjacent (stride_head == S)
    uint32_t rows_contig;       // token rows adjacent too (stride_token == Hk * S)
    uint32_t tables_bytes;      // shared bytes of the staged ragged tables (x128)
    uint32_t stage_bytes, q_off, k_off, f_off, meta_off;  // stage layout
    uint32_t slices;            // head slices per (token, pair group)
    uint32_t items;             // (Hq + Hk) * S / 16 (register-staged kernel)
    uint64_t wait_ns;           // limit of every mbarrier wait of the pipeline
    FastDiv ps_div;             // division by page_size
    FastDiv g_div, sl_div;      // by the 8-pair groups per head and the head slices
    FastDiv half_div;           // by the pairs per head (S / 2)
};

__device__ __forceinline__ uint32_t section_of(const GqaArgs& a, uint32_t k) {
    return k < a.sec0 ? 0u : (k < a.sec01 ? 1u : 2u);
}

// Whether mrope position row r supplies any pair (its section is not empty).
__device__ __forceinline__ bool section_used(const GqaArgs& a, uint32_t r) {
    return r == 0 ? a.sec0 > 0u : (r == 1 ? a.sec01 > a.sec0 : (a.S >> 1) > a.sec01);
}

struct TokMeta {
    int64_t kbase;  // element offset of the K row (head 0), -1: not written
    uint32_t qok;   // RoPE positions valid: query and key rows may be written
    uint32_t pad;
};

// WITHHOLD (test builds only): the first group of every CTA is announced on
// its stage barrier but none of its copies is issued, so the consumers' wait
// for that stage runs into its limit.
template <bool WITHHOLD>
__device__ __forceinline__ void producer(const GqaArgs& a, uint64_t* full, uint64_t* empty,
                                         const uint32_t* s_off, const uint32_t* s_clen,
                                         unsigned char* stages) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t row_bytes = a.S * 2u;       // a query row
    const uint32_t krow_bytes = a.S * a.kesz;  // a key row
    uint32_t it = 0;
    for (uint32_t g = blockIdx.x; g < a.groups; g += gridDim.x, ++it) {
        const uint32_t s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        // With position_ids the slot resolution takes two dependent loads
        // (position, then page); resolving before waiting for the stage hides
        // them under the consumers' work.  With slot positions (one load) the
        // wait comes first: that order measured faster there.
        const bool early = a.mode != 0;
        if (!early && it >= (uint32_t)kStages && !mbar_wait(&empty[s], ph ^ 1u, a.wait_ns)) {
            if (lane == 0) flag(a.err_flags, KVW_ERR_TIMEOUT);
            break;
        }
        const uint32_t t0 = g * a.tpb;
        const uint32_t ntok = min(a.tpb, a.T - t0);
        uint64_t p = 0;  // RoPE position: the slot position, or position_ids[t]
        int64_t kbase = -1;
        uint32_t qok = 0, bytes = 0;
        if (lane < ntok) {
            const uint32_t t = t0 + lane;
            const uint32_t b = find_request(s_off, a.B, t);
            const uint64_t pos = (uint64_t)s_clen[b] + (t - s_off[b]);
            p = a.mode == 0 ? pos : (uint64_t)__ldg(a.position_ids + t);
            qok = p < a.freqs_rows;
            if (!qok) {
                flag(a.err_flags, KVW_ERR_POSITION);
            } else {
                kbase = slot_row(a.page_table, a.max_pages, a.num_pages, a.ps_div, a.s_page,
                                 a.s_token, a.layer_off, b, pos);
                if (kbase < 0) flag(a.err_flags, KVW_ERR_PAGE);
                bytes += a.S * 4u;  // the freqs row
                if (kbase >= 0) bytes += a.Hk * krow_bytes;
            }
        }
        if (early && it >= (uint32_t)kStages && !mbar_wait(&empty[s], ph ^ 1u, a.wait_ns)) {
            if (lane == 0) flag(a.err_flags, KVW_ERR_TIMEOUT);
            break;
        }
        unsigned char* st = stages + (size_t)s * a.stage_bytes;
        TokMeta* meta = reinterpret_cast<TokMeta*>(st + a.meta_off);
        if (lane < ntok) {
            meta[lane].kbase = kbase;
            meta[lane].qok = qok;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
        const uint32_t qbytes = ntok * a.Hq * row_bytes;
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes + qbytes);
        __syncwarp();
        if (WITHHOLD && it == 0) continue;
        if (lane == 0 && qbytes)
            bulk_load(st + a.q_off, a.q_in + (uint64_t)t0 * a.Hq * a.S, qbytes, &full[s]);
        // K rows: one copy per run of tokens whose rows are adjacent in the
        // cache (consecutive slots of a page, dense token rows); freqs rows:
        // one copy per run of consecutive positions when positions are the
        // slot positions.  Runs cut the number of copies per group from
        // about 2 x TPB to a few.
        const int64_t kprev = __shfl_up_sync(0xffffffffu, kbase, 1);
        const bool kcont = a.rows_contig && lane > 0 && lane < ntok && qok && kbase >= 0 &&
                           kprev >= 0 && kbase == kprev + a.s_token;
        const uint32_t kstarts = __ballot_sync(0xffffffffu, lane < ntok && qok && kbase >= 0 && !kcont);
        const uint64_t pprev = __shfl_up_sync(0xffffffffu, p, 1);
        const uint32_t qok_mask = __ballot_sync(0xffffffffu, lane < ntok && qok);
        const bool fcont = a.mode == 0 && lane > 0 && lane < ntok && qok &&
                           ((qok_mask >> (lane - 1)) & 1u) && p == pprev + 1;
        const uint32_t fstarts = __ballot_sync(0xffffffffu, lane < ntok && qok && !fcont);
        if (lane < ntok && qok) {
            if (kbase >= 0 && !kcont) {
                unsigned char* kdst = st + a.k_off + (size_t)lane * a.Hk * krow_bytes;
                const unsigned char* ksrc = a.cache + kbase * a.kesz;
                if (a.rows_contig) {
                    uint32_t n = 1;  // run length: up to the next run start
                    while (lane + n < ntok && ((kstarts >> (lane + n)) & 1u) == 0u &&
                           ((qok_mask >> (lane + n)) & 1u) && meta[lane + n].kbase >= 0)
                        ++n;
                    bulk_load(kdst, ksrc, n * a.Hk * krow_bytes, &full[s]);
                } else if (a.heads_contig) {
                    bulk_load(kdst, ksrc, a.Hk * krow_bytes, &full[s]);
                } else {
                    for (uint32_t h = 0; h < a.Hk; ++h)
                        bulk_load(kdst + h * krow_bytes, ksrc + (int64_t)h * a.s_head * a.kesz,
                                  krow_bytes, &full[s]);
                }
            }
            if (!fcont) {  // one copy per run of consecutive positions (always 1 with ids)
                uint32_t n = 1;
                while (lane + n < ntok && ((fstarts >> (lane + n)) & 1u) == 0u &&
                       ((qok_mask >> (lane + n)) & 1u))
                    ++n;
                bulk_load(st + a.f_off + (size_t)lane * a.S * 4u, a.freqs + p * a.S, n * a.S * 4u,
                          &full[s]);
            }
        }
    }
    // Do not leave the CTA with copies in flight: wait for the stages issued last.
    if (lane == 0) {
        for (uint32_t j = it > (uint32_t)kStages ? it - kStages : 0u; j < it; ++j)
            if (!mbar_wait(&full[j % kStages], (j / kStages) & 1u, a.wait_ns))
                flag(a.err_flags, KVW_ERR_TIMEOUT);
    }
}

template <bool INTERLEAVED, bool FP8K>
__device__ __forceinline__ void consumer(const GqaArgs& a, uint64_t* full, uint64_t* empty,
                                         const unsigned char* stages) {
    const uint32_t tid = threadIdx.x, lane = tid & 31u;
    const uint32_t G = a.S >> 4;  // 8-pair groups per head
    const uint32_t H = a.Hq + a.Hk;
    const uint32_t hps = (H + a.slices - 1) / a.slices;
    const uint32_t units = a.tpb * G * a.slices;
    // element offsets of the two 8-element vectors of pair group m in a head row
    uint32_t it = 0;
    for (uint32_t g = blockIdx.x; g < a.groups; g += gridDim.x, ++it) {
        const uint32_t s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        if (!mbar_wait(&full[s], ph, a.wait_ns)) {
            if (lane == 0) flag(a.err_flags, KVW_ERR_TIMEOUT);
            return;
        }
        const unsigned char* st = stages + (size_t)s * a.stage_bytes;
        const TokMeta* meta = reinterpret_cast<const TokMeta*>(st + a.meta_off);
        const uint32_t t0 = g * a.tpb;
        const uint32_t ntok = min(a.tpb, a.T - t0);
        for (uint32_t w = tid; w < units; w += kConsumers) {
            const uint32_t rest = fast_div(w, a.g_div);
            const uint32_t m = w - rest * G;
            const uint32_t u = fast_div(rest, a.sl_div);
            const uint32_t sl = rest - u * a.slices;
            if (u >= ntok) continue;
            const TokMeta tm = meta[u];
            if (!tm.qok) continue;
            const uint32_t h_begin = sl * hps;
            const uint32_t h_end = min(H, h_begin + hps);
            if (h_begin >= h_end) continue;
            // (cos, sin) of pairs 8m .. 8m+7
            float c[8], sn[8];
            const float* frow = reinterpret_cast<const float*>(st + a.f_off) + (size_t)u * a.S;
            {
                // The 8 lanes of a quarter-warp (m = 0..7) would read their
                // float4 q at 64 m + 16 q: 2 bank groups, 4-way conflicts.
                // Lane m reads them rotated by r = m / 2 (8 distinct bank
                // groups per load) and rotates them back with selects.
                const float4* f4 = reinterpret_cast<const float4*>(frow + 16u * m);
                const uint32_t r = (m >> 1) & 3u;
                float4 t[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) t[q] = f4[(q + r) & 3u];
                if (r & 1u) {  // rotate right by one
                    const float4 x = t[3];
                    t[3] = t[2];
                    t[2] = t[1];
                    t[1] = t[0];
                    t[0] = x;
                }
                if (r & 2u) {  // rotate right by two
                    float4 x = t[0];
                    t[0] = t[2];
                    t[2] = x;
                    x = t[1];
                    t[1] = t[3];
                    t[3] = x;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v = t[q];
                    c[2 * q] = v.x;
                    sn[2 * q] = v.y;
                    c[2 * q + 1] = v.z;
                    sn[2 * q + 1] = v.w;
                }
            }
            const uint32_t e0 = INTERLEAVED ? 16u * m : 8u * m;
            const uint32_t e1 = INTERLEAVED ? 16u * m + 8u : (a.S >> 1) + 8u * m;
            for (uint32_t h = h_begin; h < h_end; ++h) {
                const bool is_q = h < a.Hq;
                if (!is_q && tm.kbase < 0) break;
                float va[8], vb[8], ya[8], yb[8];
                if (!FP8K) {
                    // Interleaved: the two vectors of group m are adjacent, so
                    // the 8 lanes of a quarter-warp (m = 0..7) would read
                    // 16-byte slots 2m and hit each bank group twice; groups
                    // 4..7 read their second vector first, which spreads the
                    // 8 slots of every load over all 32 banks (2% faster with
                    // a bf16 K cache; the FP8 K build measured slower with it).
                    const uint16_t* src =
                        is_q ? reinterpret_cast<const uint16_t*>(st + a.q_off) +
                                   ((size_t)u * a.Hq + h) * a.S
                             : reinterpret_cast<const uint16_t*>(st + a.k_off) +
                                   ((size_t)u * a.Hk + (h - a.Hq)) * a.S;
                    const bool swz = INTERLEAVED && (m & 4u);
                    const uint4 ra = *reinterpret_cast<const uint4*>(src + (swz ? e1 : e0));
                    const uint4 rb = *reinterpret_cast<const uint4*>(src + (swz ? e0 : e1));
                    unpack8(swz ? rb : ra, va);
                    unpack8(swz ? ra : rb, vb);
                } else if (is_q) {
                    const uint16_t* src =
                        reinterpret_cast<const uint16_t*>(st + a.q_off) + ((size_t)u * a.Hq + h) * a.S;
                    unpack8(*reinterpret_cast<const uint4*>(src + e0), va);
                    unpack8(*reinterpret_cast<const uint4*>(src + e1), vb);
                } else {
                    const unsigned char* src =
                        st + a.k_off + ((size_t)u * a.Hk + (h - a.Hq)) * a.S * a.kesz;
                    load_k8<FP8K>(src + e0 * a.kesz, va, a.kscale);
                    load_k8<FP8K>(src + e1 * a.kesz, vb, a.kscale);
                }
                if (INTERLEAVED) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        rope_pair(va[2 * q], va[2 * q + 1], c[q], sn[q], ya[2 * q], ya[2 * q + 1]);
                        rope_pair(vb[2 * q], vb[2 * q + 1], c[q + 4], sn[q + 4], yb[2 * q],
                                  yb[2 * q + 1]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q) rope_pair(va[q], vb[q], c[q], sn[q], ya[q], yb[q]);
                }
                if (is_q) {
                    uint16_t* dst = a.q_out + ((uint64_t)(t0 + u) * a.Hq + h) * a.S;
                    st_stream(reinterpret_cast<uint4*>(dst + e0), pack8_bf16(ya));
                    st_stream(reinterpret_cast<uint4*>(dst + e1), pack8_bf16(yb));
                } else {
                    unsigned char* dst =
                        a.cache + (tm.kbase + (int64_t)(h - a.Hq) * a.s_head) * a.kesz;
                    store_k8<FP8K>(dst + e0 * a.kesz, ya, a.kscale);
                    store_k8<FP8K>(dst + e1 * a.kesz, yb, a.kscale);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// CTAs per SM: one for a bf16 K cache; two for an E4M3 K cache, whose
// consumers spend more instructions per byte (decode, re-encode) and keep up
// better with two CTAs' warps interleaved (stages sized for two CTAs).
template <bool FP8K>
constexpr int kCtasPerSm = FP8K ? 2 : 1;

template <bool INTERLEAVED, bool FP8K, bool WITHHOLD>
__global__ void __launch_bounds__(kThreads, kCtasPerSm<FP8K>) qk_rope_kernel(const GqaArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStages;
    uint32_t* s_off = reinterpret_cast<uint32_t*>(smem + 128);
    uint32_t* s_clen = s_off + a.B + 1;
    unsigned char* stages = smem + 128 + a.tables_bytes;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init_fence();
    }
    // the barrier inside also publishes the mbarrier initialisation
    if (!stage_ragged(a.offsets, a.cache_lengths, a.B, a.T, s_off, s_clen)) {
        if (threadIdx.x == 0) flag(a.err_flags, KVW_ERR_OFFSETS);
        return;
    }
    if (threadIdx.x >= (unsigned)kConsumers)
        producer<WITHHOLD>(a, full, empty, s_off, s_clen, stages);
    else
        consumer<INTERLEAVED, FP8K>(a, full, empty, stages);
}

template <bool INTERLEAVED, bool FP8K, bool WITHHOLD = false>
cudaError_t launch(const GqaArgs& a, size_t smem, cudaStream_t stream) {
    constexpr auto k = qk_rope_kernel<INTERLEAVED, FP8K, WITHHOLD>;
    uint64_t cap = 0;
    const cudaError_t e = wave_ctas<k>(kThreads, smem, cap);
    if (e != cudaSuccess) return e;
    if (cap == 0) return cudaErrorInvalidConfiguration;
    const uint32_t grid = (uint32_t)(a.groups < cap ? a.groups : cap);
    k<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------
// Register-staged variant, used for mrope.  With three position rows per
// token the pipelined kernel would need three small freqs copies per token
// (or a composed row built by the producer warp), and both measured slower
// than this.  The CTA has one thread per 8-pair item of a token (rounded up
// to warps) and is persistent: it stages the ragged tables once, then walks
// groups of TPB tokens.  For the group in hand, every thread loads its query
// vectors and (slot rows already known) its key vectors; while those loads
// are in flight it prepares the next group into the other half of a
// double-buffered shared area -- slot rows and position checks (one thread
// per token) and the composed (cos, sin) row of each token (all threads,
// one pair each) -- then rotates and stores the group in hand.
// Composed (cos, sin) rows are stored swizzled: float4 q (pairs 8m + 2q and
// 8m + 2q + 1) of pair group m sits in slot (q + m / 2) mod 4 of the group's
// four, so when the 8 lanes of a quarter-warp (m = 0..7) read their float4 q
// they touch 8 different 16-byte bank groups instead of 2.
__device__ __forceinline__ uint32_t cs_slot(uint32_t m, uint32_t q) {
    return 16u * m + 4u * ((q + (m >> 1)) & 3u);
}

template <int TPB>
struct StagedSmem {
    float cs[2][TPB][kMaxHead];  // composed (cos, sin) per pair, swizzled (cs_slot)
    int64_t kbase[2][TPB];       // slot row of each token (-1: no page)
    int bad[2][TPB];             // a RoPE position of the token is out of range
};

template <int TPB>
__device__ __forceinline__ void staged_prepare(const GqaArgs& a, const uint32_t* s_off,
                                               const uint32_t* s_clen, StagedSmem<TPB>& sm,
                                               uint32_t buf, uint32_t group) {
    const uint32_t t_begin = group * TPB;
    const uint32_t i = threadIdx.x;
    if (i < TPB) {
        const uint32_t t = t_begin + i;
        int64_t base = -1;
        int bad = 0;
        if (t < a.T) {
            const uint32_t b = find_request(s_off, a.B, t);
            const uint64_t pos = (uint64_t)s_clen[b] + (t - s_off[b]);
            base = slot_row(a.page_table, a.max_pages, a.num_pages, a.ps_div, a.s_page,
                            a.s_token, a.layer_off, b, pos);
            if (a.mode == 0) {
                bad = pos >= a.freqs_rows;
            } else if (a.mode == 1) {
                bad = __ldg(a.position_ids + t) >= a.freqs_rows;
            } else {
                for (uint32_t r = 0; r < 3; ++r)
                    if (section_used(a, r) &&
                        __ldg(a.position_ids + (uint64_t)r * a.T + t) >= a.freqs_rows)
                        bad = 1;
            }
        }
        sm.kbase[buf][i] = base;
        sm.bad[buf][i] = bad;
    }
    const uint32_t half = a.S >> 1;
    for (uint32_t idx = threadIdx.x; idx < TPB * half; idx += blockDim.x) {
        const uint32_t u = fast_div(idx, a.half_div), k = idx - u * half;
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
        if (p < a.freqs_rows) cs = __ldg(reinterpret_cast<const float2*>(a.freqs + p * a.S) + k);
        *reinterpret_cast<float2*>(&sm.cs[buf][u][cs_slot(k >> 3, (k >> 1) & 3u) + 2u * (k & 1u)]) = cs;
    }
}

template <bool INTERLEAVED, int TPB, bool FP8K>
__global__ void __launch_bounds__(1024) qk_rope_staged_kernel(const GqaArgs a) {
    extern __shared__ uint32_t s_dyn[];
    uint32_t* s_off = s_dyn;
    uint32_t* s_clen = s_dyn + a.B + 1;
    __shared__ __align__(16) StagedSmem<TPB> sm;

    const uint32_t groups = a.S >> 4;  // items per head
    const uint32_t i = threadIdx.x;
    const bool has_item = i < a.items;
    const uint32_t h = has_item ? i / groups : 0u;
    const uint32_t m = has_item ? i % groups : 0u;
    const bool is_q = has_item && h < a.Hq;
    // element offsets of the two vectors of this item inside a head row
    const uint32_t e0 = INTERLEAVED ? 16u * m : 8u * m;
    const uint32_t e1 = INTERLEAVED ? 16u * m + 8u : (a.S >> 1) + 8u * m;

    if (!stage_ragged(a.offsets, a.cache_lengths, a.B, a.T, s_off, s_clen)) {
        if (threadIdx.x == 0) flag(a.err_flags, KVW_ERR_OFFSETS);
        return;
    }
    const uint32_t ngroups = (a.T + TPB - 1) / TPB;
    uint32_t g = blockIdx.x;
    if (g >= ngroups) return;
    staged_prepare<TPB>(a, s_off, s_clen, sm, 0, g);
    __syncthreads();

    for (uint32_t buf = 0; g < ngroups; g += gridDim.x, buf ^= 1u) {
        const uint32_t t_begin = g * TPB;
        // query and key data of the group in hand
        uint4 xa[TPB], xb[TPB];
#pragma unroll
        for (int u = 0; u < TPB; ++u) {
            xa[u] = make_uint4(0, 0, 0, 0);
            xb[u] = xa[u];
            const uint32_t t = t_begin + u;
            if (t >= a.T || sm.bad[buf][u]) continue;
            if (is_q) {
                const uint16_t* row = a.q_in + ((uint64_t)t * a.Hq + h) * a.S;
                xa[u] = ld_stream(reinterpret_cast<const uint4*>(row + e0));
                xb[u] = ld_stream(reinterpret_cast<const uint4*>(row + e1));
            } else if (has_item && sm.kbase[buf][u] >= 0) {
                const unsigned char* row =
                    a.cache + (sm.kbase[buf][u] + (int64_t)(h - a.Hq) * a.s_head) * a.kesz;
                if (FP8K) {  // 8 codes per vector: kept in .x/.y
                    const uint2 va8 = *reinterpret_cast<const uint2*>(row + e0);
                    const uint2 vb8 = *reinterpret_cast<const uint2*>(row + e1);
                    xa[u] = make_uint4(va8.x, va8.y, 0, 0);
                    xb[u] = make_uint4(vb8.x, vb8.y, 0, 0);
                } else {
                    xa[u] = *reinterpret_cast<const uint4*>(row + 2 * e0);
                    xb[u] = *reinterpret_cast<const uint4*>(row + 2 * e1);
                }
            }
        }
        // the next group, while those loads are in flight
        if (g + gridDim.x < ngroups) staged_prepare<TPB>(a, s_off, s_clen, sm, buf ^ 1u, g + gridDim.x);
        if (i < TPB && t_begin + i < a.T) {
            if (sm.bad[buf][i])
                flag(a.err_flags, KVW_ERR_POSITION);
            else if (sm.kbase[buf][i] < 0)
                flag(a.err_flags, KVW_ERR_PAGE);
        }
        if (has_item) {
#pragma unroll
            for (int u = 0; u < TPB; ++u) {
                const uint32_t t = t_begin + u;
                if (t >= a.T || sm.bad[buf][u]) continue;
                if (!is_q && sm.kbase[buf][u] < 0) continue;
                const float* row = sm.cs[buf][u];
                const float4 c0 = *reinterpret_cast<const float4*>(row + cs_slot(m, 0));
                const float4 c1 = *reinterpret_cast<const float4*>(row + cs_slot(m, 1));
                const float4 c2 = *reinterpret_cast<const float4*>(row + cs_slot(m, 2));
                const float4 c3 = *reinterpret_cast<const float4*>(row + cs_slot(m, 3));
                const float c[8] = {c0.x, c0.z, c1.x, c1.z, c2.x, c2.z, c3.x, c3.z};
                const float s[8] = {c0.y, c0.w, c1.y, c1.w, c2.y, c2.w, c3.y, c3.w};
                float va[8], vb[8], ya[8], yb[8];
                if (FP8K && !is_q) {
                    unpack8_e4m3(make_uint2(xa[u].x, xa[u].y), va);
                    unpack8_e4m3(make_uint2(xb[u].x, xb[u].y), vb);
                    if (a.kscale != 1.0f) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            va[q] = __fmul_rn(va[q], a.kscale);
                            vb[q] = __fmul_rn(vb[q], a.kscale);
                        }
                    }
                } else {
                    unpack8(xa[u], va);
                    unpack8(xb[u], vb);
                }
                if (INTERLEAVED) {  // pairs (va0,va1) (va2,va3) .. (vb6,vb7)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        rope_pair(va[2 * q], va[2 * q + 1], c[q], s[q], ya[2 * q], ya[2 * q + 1]);
                        rope_pair(vb[2 * q], vb[2 * q + 1], c[q + 4], s[q + 4], yb[2 * q],
                                  yb[2 * q + 1]);
                    }
                } else {  // pairs (va[q], vb[q])
#pragma unroll
                    for (int q = 0; q < 8; ++q) rope_pair(va[q], vb[q], c[q], s[q], ya[q], yb[q]);
                }
                if (is_q) {
                    uint16_t* row = a.q_out + ((uint64_t)t * a.Hq + h) * a.S;
                    st_stream(reinterpret_cast<uint4*>(row + e0), pack8_bf16(ya));
                    st_stream(reinterpret_cast<uint4*>(row + e1), pack8_bf16(yb));
                } else {
                    unsigned char* row =
                        a.cache + (sm.kbase[buf][u] + (int64_t)(h - a.Hq) * a.s_head) * a.kesz;
                    store_k8<FP8K>(row + e0 * a.kesz, ya, a.kscale);
                    store_k8<FP8K>(row + e1 * a.kesz, yb, a.kscale);
                }
            }
        }
        __syncthreads();  // next group's tables visible; this group's no longer read
    }
}

template <bool INTERLEAVED, int TPB, bool FP8K>
cudaError_t launch_staged(const GqaArgs& a, uint32_t threads, size_t smem, cudaStream_t stream) {
    constexpr auto k = qk_rope_staged_kernel<INTERLEAVED, TPB, FP8K>;
    uint64_t wave = 0;
    const cudaError_t e = wave_ctas<k>((int)threads, smem, wave);
    if (e != cudaSuccess) return e;
    if (wave == 0) return cudaErrorInvalidConfiguration;
    const uint64_t groups = (a.T + TPB - 1) / TPB;
    k<<<(uint32_t)(groups < wave ? groups : wave), threads, smem, stream>>>(a);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvw

namespace kvw {
namespace {

// Validation, sizing and launch.  `withhold` (test builds only) launches the
// pipelined kernel with its first group's copies withheld; `wait_ns` bounds
// every wait of the pipeline.
int qk_entry(const void* q_proj, const uint32_t* input_row_offsets, uint32_t num_batches,
             uint32_t tot_seq_len, uint32_t num_q_heads, const kvw_paged_cache_t* cache,
             const void* freqs_cis, uint32_t freqs_rows, const uint32_t* position_ids,
             int interleaved, const uint32_t* mrope_section, uint32_t layer_idx, void* output,
             uint32_t* err_flags, cudaStream_t stream, bool withhold, uint64_t wait_ns) {
    if (!cache) return KVW_EINVAL;
    if (cache->dtype != KVW_DTYPE_BF16 && cache->dtype != KVW_DTYPE_FP8_E4M3)
        return KVW_EUNSUPPORTED;
    const bool fp8 = cache->dtype == KVW_DTYPE_FP8_E4M3;
    const int64_t esz = fp8 ? 1 : 2;
    if (fp8 && !(cache->scale > 0.0f && cache->scale < 3.0e38f)) return KVW_EINVAL;
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
    if ((cache->stride_page * esz) % 16 || (cache->stride_layer * esz) % 16 ||
        (cache->stride_token * esz) % 16 || (cache->stride_head * esz) % 16 ||
        cache->stride_page <= 0 || cache->stride_token <= 0)
        return KVW_EINVAL;
    if (items == 0) return KVW_OK;

    GqaArgs a;
    a.q_in = static_cast<const uint16_t*>(q_proj);
    a.q_out = static_cast<uint16_t*>(output);
    a.cache = static_cast<unsigned char*>(cache->data);
    a.kscale = cache->scale;
    a.kesz = (uint32_t)esz;
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
    a.wait_ns = wait_ns;
    a.ps_div = make_fast_div(cache->page_size);
    a.half_div = make_fast_div(S / 2);
    a.g_div = make_fast_div(S / 16);
    a.sl_div = make_fast_div(1);
    if (withhold && a.mode == 2) return KVW_EUNSUPPORTED;  // the hook is in the pipeline only
    if (a.mode == 2) {
        const uint32_t threads = (uint32_t)((items + 31) / 32 * 32);
        const size_t smem_st = sizeof(uint32_t) * (2 * (size_t)num_batches + 1);
        // small batches: smaller groups, so that every SM gets a few of them
        int sms = 0;
        if (sm_count(sms) != cudaSuccess) return KVW_ECUDA;
        int tpb = 4;
        while (tpb > 1 && (uint64_t)(tot_seq_len + tpb - 1) / tpb < (uint64_t)sms * 4) tpb >>= 1;
        cudaError_t es;
        auto pick = [&](auto il, auto f8) {
            constexpr bool IL = decltype(il)::value, F8 = decltype(f8)::value;
            return tpb == 4 ? launch_staged<IL, 4, F8>(a, threads, smem_st, stream)
                 : tpb == 2 ? launch_staged<IL, 2, F8>(a, threads, smem_st, stream)
                            : launch_staged<IL, 1, F8>(a, threads, smem_st, stream);
        };
        using T_ = std::true_type;
        using F_ = std::false_type;
        es = interleaved ? (fp8 ? pick(T_{}, T_{}) : pick(T_{}, F_{}))
                         : (fp8 ? pick(F_{}, T_{}) : pick(F_{}, F_{}));
        return es == cudaSuccess ? KVW_OK : KVW_ECUDA;
    }
    a.heads_contig = cache->stride_head == (int64_t)S ? 1u : 0u;
    a.rows_contig = a.heads_contig && cache->stride_token == (int64_t)a.Hk * S ? 1u : 0u;

    // shared memory: barriers | ragged tables | kStages x (q | k | freqs | meta)
    const uint32_t tables = (uint32_t)(((2ull * num_batches + 1) * 4 + 127) / 128 * 128);
    const uint64_t per_tok = (uint64_t)num_q_heads * S * 2 + (uint64_t)a.Hk * S * esz +
                             (uint64_t)S * 4 +
                             sizeof(TokMeta);
    int optin = 0, sms = 0;
    if (smem_optin(optin) != cudaSuccess || sm_count(sms) != cudaSuccess) return KVW_ECUDA;
    // shared memory of one CTA: an SM holds 1 (bf16 K) or 2 (E4M3 K) CTAs, each
    // with 1 KiB reserved by the runtime
    const uint64_t ctas = fp8 ? 2 : 1;
    const uint64_t budget = ((uint64_t)optin + 1024) / ctas - 1024 - 128 - tables - kStages * 1024;
    uint64_t tpb_max = budget / (kStages * per_tok);
    if (tpb_max > kMaxTPB) tpb_max = kMaxTPB;
    // small batches: spread the groups over all SMs
    const uint64_t spread = (tot_seq_len + (uint64_t)sms - 1) / sms;
    if (tpb_max > spread) tpb_max = spread;
    if (tpb_max == 0) return KVW_EUNSUPPORTED;
    // Tokens per group: the consumers split a group into tpb * G * slices
    // units (one per thread), each rotating ceil(H / slices) heads.  The use
    // of a split counts idle threads and the largest slice against the
    // average one (for 40 heads of 128: 10 tokens x 3 slices use 0.89 of the
    // consumers, 11 tokens x 2 slices 0.69).  Larger groups cost less
    // producer work per token, so take the largest group whose use is at
    // least 0.85, else the group size of the best use; among equal uses, the
    // largest group that leaves no consumer thread idle (40 heads of 128 with
    // an E4M3 K cache: 4 tokens x 12 slices rather than 5 x 9, which idles 24
    // of 384 threads; 2.5% faster in a same-box A/B).
    const uint32_t G_ = S / 16, H_ = num_q_heads + a.Hk;
    uint64_t tpb = tpb_max;
    double best = -1.0;
    bool best_full = false;
    for (uint64_t c = tpb_max; c >= 1; --c) {
        uint64_t sl = kConsumers / (c * G_);
        if (sl < 1) sl = 1;
        if (sl > H_) sl = H_;
        const uint64_t units = c * G_ * sl;
        const uint64_t passes = (units + kConsumers - 1) / kConsumers;
        const uint64_t hps = (H_ + sl - 1) / sl;
        const double use = (double)units / (double)(passes * kConsumers) *
                           ((double)H_ / (double)sl) / (double)hps;
        if (use >= 0.85) {
            tpb = c;
            break;
        }
        const bool full = units == passes * kConsumers;
        if (use > best + 1e-9 || (use > best - 1e-9 && full && !best_full)) {
            if (use > best) best = use;
            best_full = full;
            tpb = c;
        }
    }
    a.tpb = (uint32_t)tpb;
    a.groups = (uint32_t)((tot_seq_len + tpb - 1) / tpb);
    a.tables_bytes = tables;
    auto up16 = [](uint64_t x) { return (uint32_t)((x + 15) / 16 * 16); };
    a.q_off = 0;
    a.k_off = up16(tpb * num_q_heads * S * 2);
    a.f_off = a.k_off + up16(tpb * a.Hk * S * esz);
    a.meta_off = a.f_off + up16(tpb * S * 4);
    a.stage_bytes = (uint32_t)((a.meta_off + tpb * sizeof(TokMeta) + 127) / 128 * 128);
    const uint32_t G = S / 16;
    a.slices = (uint32_t)(kConsumers / (tpb * G));
    if (a.slices < 1) a.slices = 1;
    if (a.slices > num_q_heads + a.Hk) a.slices = num_q_heads + a.Hk;
    a.sl_div = make_fast_div(a.slices);
    const size_t smem = 128 + (size_t)tables + (size_t)kStages * a.stage_bytes;
    if (smem > (size_t)optin) return KVW_EUNSUPPORTED;
    cudaError_t e;
#ifdef KVW_TEST_HOOKS
    if (withhold)
        e = interleaved ? (fp8 ? launch<true, true, true>(a, smem, stream)
                               : launch<true, false, true>(a, smem, stream))
                        : (fp8 ? launch<false, true, true>(a, smem, stream)
                               : launch<false, false, true>(a, smem, stream));
    else
#else
    if (withhold) return KVW_EUNSUPPORTED;
#endif
        e = interleaved ? (fp8 ? launch<true, true>(a, smem, stream)
                               : launch<true, false>(a, smem, stream))
                        : (fp8 ? launch<false, true>(a, smem, stream)
                               : launch<false, false>(a, smem, stream));
    return e == cudaSuccess ? KVW_OK : KVW_ECUDA;
}

}  // namespace
}  // namespace kvw

extern "C" int kvw_qk_rope_paged_ragged(const void* q_proj, const uint32_t* input_row_offsets,
                                        uint32_t num_batches, uint32_t tot_seq_len,
                                        uint32_t num_q_heads, const kvw_paged_cache_t* cache,
                                        const void* freqs_cis, uint32_t freqs_rows,
                                        const uint32_t* position_ids, int interleaved,
                                        const uint32_t* mrope_section, uint32_t layer_idx,
                                        void* output, uint32_t* err_flags, cudaStream_t stream) {
    return kvw::qk_entry(q_proj, input_row_offsets, num_batches, tot_seq_len, num_q_heads, cache,
                         freqs_cis, freqs_rows, position_ids, interleaved, mrope_section,
                         layer_idx, output, err_flags, stream, false, kvw::kWaitLimitNs);
}

#ifdef KVW_TEST_HOOKS
// Test builds only (compiled with -DKVW_TEST_HOOKS into a separate library;
// the product library has no such symbol): the pipelined GQA kernel with the
// first group of every CTA announced on its stage barrier but never copied,
// and every wait bounded by `wait_ns`, so the consumers' wait for that stage
// runs out, KVW_ERR_TIMEOUT is set and the kernel returns.
extern "C" int kvw_test_qk_rope_withheld_stage(
    const void* q_proj, const uint32_t* input_row_offsets, uint32_t num_batches,
    uint32_t tot_seq_len, uint32_t num_q_heads, const kvw_paged_cache_t* cache,
    const void* freqs_cis, uint32_t freqs_rows, const uint32_t* position_ids, int interleaved,
    uint32_t layer_idx, void* output, uint32_t* err_flags, cudaStream_t stream,
    uint64_t wait_ns) {
    return kvw::qk_entry(q_proj, input_row_offsets, num_batches, tot_seq_len, num_q_heads, cache,
                         freqs_cis, freqs_rows, position_ids, interleaved, nullptr, layer_idx,
                         output, err_flags, stream, true, wait_ns);
}
#endif
