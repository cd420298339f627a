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
    FastDiv ps_div;    // division by page_size
    uint64_t wait_ns;  // limit of every mbarrier wait
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

// row_base in two halves, so that the page-table load can be issued a step
// before its value is needed: row_lookup finds the request and loads the page
// id of output row r, row_resolve checks the page and forms the offset.
struct RowLookup {
    uint32_t page;
    int64_t off;  // cache elements within the page (layer and token); < 0: no row
};
__device__ __forceinline__ RowLookup row_lookup(const GatherArgs& a, const uint32_t* s_off,
                                                uint32_t r) {
    RowLookup l{KVW_PAGE_UNMAPPED, -1};
    if (r >= a.rows) return l;
    const uint32_t b = find_request(s_off, a.B, r);
    const uint32_t pos = r - s_off[b];
    const uint32_t pidx = fast_div(pos, a.ps_div);
    if (pidx < a.max_pages) l.page = __ldg(a.page_table + (uint64_t)b * a.max_pages + pidx);
    l.off = a.layer_off + (int64_t)(pos - pidx * a.page_size) * a.s_token;
    return l;
}
__device__ __forceinline__ int64_t row_resolve(const GatherArgs& a, const RowLookup& l) {
    if (l.off < 0) return -1;
    if (l.page >= a.num_pages) {
        flag(a.err_flags, KVW_ERR_PAGE);
        return -1;
    }
    return (int64_t)l.page * a.s_page + l.off;
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
// are maxima of magnitudes in each lane and one warp redux per row, and the
// scale and its reciprocal are computed in registers -- no shared-memory
// reduction and no block barrier after the offsets are staged.  The source
// rows reach the warp through shared memory: each warp runs its own ring of
// kDynStages stages of kDynRows rows, one bulk asynchronous copy per row
// completing on the stage's mbarrier.  A step reads its stage twice, once for
// the maxima and once for the codes, so that no piece is held in registers
// across the reductions (the register count allows 3 CTAs per SM); then the
// warp refills the stage with its step kDynStages ahead.  The page ids of
// that step's rows (lane q < kDynRows: request by binary search, page from
// the page table) were loaded a step earlier, so the refill waits on no load.
// Values that are bf16 numbers (a bf16 cache, or E4M3 codes at cache scale 1)
// divide by the scale through div_refined; others through the IEEE divide.
constexpr uint32_t kDynRows = 4;

// Bit pattern of the largest magnitude among 8 E4M3 cache values times the
// cache scale, as an fp32 (non-negative floats order like their bit
// patterns).  The sign-cleared codes order like the magnitudes, so a per-byte
// unsigned max finds it; a NaN (code 0x7F) falls back to the float maximum,
// which ignores it, as the reference maximum does.
__device__ __forceinline__ uint32_t e4m3_piece_max_bits(const uint4& raw, float cache_scale) {
    const uint32_t acc = __vmaxu4(raw.x & 0x7f7f7f7fu, raw.y & 0x7f7f7f7fu);
    const uint32_t m = max(max(acc & 0xffu, (acc >> 8) & 0xffu), max((acc >> 16) & 0xffu, acc >> 24));
    if (m != 0x7fu) {
        const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(m), __NV_E4M3);
        const float f = __half2float(__half(h));
        return __float_as_uint(cache_scale == 1.0f ? f : __fmul_rn(f, cache_scale));
    }
    float v[8];
    to_f32<true>(raw, cache_scale, v);
    float f = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) f = fmaxf(f, fabsf(v[e]));
    return __float_as_uint(f);
}

// Per-halfword maximum magnitudes of two bf16 pairs, in bits 0-14 of each
// half (bit 15 is the xor of the signs, not used).  A NaN is passed over when
// the other operand is a number, so maxima started from zero ignore NaNs, as
// the reference maximum does.
__device__ __forceinline__ uint32_t max_abs2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t halves_max(uint32_t acc, const uint4& w) {
    return max_abs2(acc, max_abs2(max_abs2(w.x, w.y), max_abs2(w.z, w.w)));
}

// 8 bf16 values -> the E4M3 codes of value / sc (y = RN(1/sc); see
// div_refined), the sign bit of each value or-ed into its code, which keeps
// the sign of -0 (a zero quotient comes out +0) and changes no other code.
// The fast path runs div_refined on fp32 pairs: the packed multiply and fused
// multiply-adds round each component exactly as the scalar ones, and x - q0 s
// is formed as fma(q0, -s, x).
__device__ __forceinline__ uint2 quantize_bf16_piece(const uint4& w, float sc, float y, bool fast) {
    float v[8];
    unpack8(w, v);
    if (fast) {
        const float2 ns2 = make_float2(-sc, -sc), y2 = make_float2(y, y);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float2 x2 = make_float2(v[e], v[e + 1]);
            const float2 q0 = __fmul2_rn(x2, y2);
            const float2 r = __ffma2_rn(q0, ns2, x2);
            const float2 q = __ffma2_rn(r, y2, q0);
            v[e] = q.x;
            v[e + 1] = q.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __fdiv_rn(v[e], sc);
    }
    uint2 c = pack8_e4m3(v);
    c.x |= __byte_perm(w.x, w.y, 0x7531u) & 0x80808080u;
    c.y |= __byte_perm(w.z, w.w, 0x7531u) & 0x80808080u;
    return c;
}

// 8 E4M3 cache codes -> the E4M3 codes of value / sc.  Values that are bf16
// numbers (cache scale 1) divide through div_refined, others through the IEEE
// divide.
__device__ __forceinline__ uint2 quantize_e4m3_piece(const uint4& raw, float cache_scale, float sc,
                                                     float y, bool fast) {
    float v[8];
    to_f32<true>(raw, cache_scale, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = fast ? div_refined(v[e], sc, y) : __fdiv_rn(v[e], sc);
    return pack8_e4m3(v);
}

// 8 bytes stored at p when `store` holds, as one predicated instruction (the
// values are computed whether or not they are stored, so no branch splits the
// code that computes them).
__device__ __forceinline__ void st_if(unsigned char* p, const uint2& v, bool store) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
        "@p st.global.v2.u32 [%1], {%2, %3};\n\t}" ::"r"((uint32_t)store),
        "l"(p), "r"(v.x), "r"(v.y)
        : "memory");
}

// A row's scale RN(amax / 448) (1 for an all-zero row): div_refined with
// RN(1/448) in [2^-100, 2^100], the IEEE divide outside.  With a fixed
// divisor, powers of two scale every step exactly, so the refinement is
// correctly rounded in that range because it is for every fp32 significand
// (all 2^23 checked on the host by tests/test_row_scale.py).
__device__ __forceinline__ float row_scale(float amax) {
    constexpr float kInv448 = 1.0f / 448.0f;
    const float q0 = __fmul_rn(amax, kInv448);
    float sc = __fmaf_rn(__fmaf_rn(-q0, 448.0f, amax), kInv448, q0);
    if (!(amax >= 0x1p-100f && amax <= 0x1p100f)) sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    return sc;
}

constexpr uint32_t kDynThreads = 256, kDynWarps = kDynThreads / 32, kDynCtasPerSm = 3;
template <bool CF8>
constexpr uint32_t kDynStages = CF8 ? 4 : 2;  // 72 KiB of stages per CTA
template <bool CF8>
constexpr uint32_t kDynRowBytes = kRow * (CF8 ? 1 : 2);
template <bool CF8>
constexpr uint32_t kDynStageBytes = kDynRows * kDynRowBytes<CF8>;

// Dynamic shared memory of gather_dynamic_kernel: the warps' stages, their
// mbarriers, then the B + 1 context offsets.
template <bool CF8>
constexpr size_t kDynStageArea = (size_t)kDynWarps * kDynStages<CF8> * kDynStageBytes<CF8>;
template <bool CF8>
size_t dyn_smem(uint32_t B) {
    return kDynStageArea<CF8> + sizeof(uint64_t) * kDynWarps * kDynStages<CF8> +
           sizeof(uint32_t) * ((size_t)B + 1);
}

// Raw bytes of 8 staged values at element `e` of a staged row.
template <bool CF8>
__device__ __forceinline__ uint4 staged_raw8(const unsigned char* row, uint32_t e) {
    if (CF8) {
        const uint2 v = *reinterpret_cast<const uint2*>(row + e);
        return make_uint4(v.x, v.y, 0, 0);
    }
    return *reinterpret_cast<const uint4*>(row + e * 2);
}

// Order this thread's shared-memory reads before later bulk copies into the
// same bytes (the copies write through the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// WITHHOLD (test builds only): the first step of every warp is announced on
// its stage barrier but not copied, so the warp's wait for it runs into its
// limit.
template <bool CF8, bool WITHHOLD = false>
__global__ void __launch_bounds__(kDynThreads, kDynCtasPerSm)
    gather_dynamic_kernel(const GatherArgs a, float* scales) {
    constexpr uint32_t S = kDynStages<CF8>, RB = kDynRowBytes<CF8>, SB = kDynStageBytes<CF8>;
    static_assert(S * kDynRows <= 32, "stage validity masks fit one word");
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t lane = threadIdx.x & 31u, wid = threadIdx.x >> 5;
    unsigned char* stages = smem + (size_t)wid * S * SB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDynStageArea<CF8>) + wid * S;
    uint32_t* s_off = reinterpret_cast<uint32_t*>(smem + kDynStageArea<CF8> +
                                                  sizeof(uint64_t) * kDynWarps * S);
    if (lane == 0) {
#pragma unroll
        for (uint32_t k = 0; k < S; ++k) mbar_init(&bars[k], 1);
        mbar_init_fence();
    }
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
    const uint32_t nwarps = gridDim.x * kDynWarps;
    const uint32_t steps = (a.rows + kDynRows - 1) / kDynRows;
    const uint32_t st0 = blockIdx.x * kDynWarps + wid;
    const int64_t esz = CF8 ? 1 : 2;
    // Copy the rows of one step (lane q < kDynRows: row q at cache element
    // `base`, or none when base < 0) into stage s; returns the rows copied.
    auto issue = [&](uint32_t s, int64_t base, bool withhold = false) -> uint32_t {
        const uint32_t valid = __ballot_sync(0xffffffffu, lane < kDynRows && base >= 0);
        if (lane == 0) mbar_arrive_expect_tx(&bars[s], __popc(valid) * RB);
        __syncwarp();
        if (((valid >> lane) & 1u) && !withhold)
            bulk_load(stages + (size_t)s * SB + lane * RB, a.cache + base * esz, RB, &bars[s]);
        return valid;
    };
    uint32_t vmask = 0;  // rows copied into stage s: bits kDynRows s ..
    RowLookup ahead;  // lane q's row of the step after the next refill
    {
        RowLookup l[S + 1];
#pragma unroll
        for (uint32_t k = 0; k <= S; ++k) {
            const uint32_t st = st0 + k * nwarps;
            l[k] = row_lookup(a, s_off, lane < kDynRows && st < steps ? st * kDynRows + lane : a.rows);
        }
#pragma unroll
        for (uint32_t k = 0; k < S; ++k)
            if (st0 + k * nwarps < steps)
                vmask |= issue(k, row_resolve(a, l[k]), WITHHOLD && k == 0) << (kDynRows * k);
        ahead = l[S];
    }
    const bool bf16_values = !CF8 || a.cache_scale == 1.0f;
    // lane l also moves the tail piece (columns 512 + 8 (l & 7) ..) of row
    // l / 8, so every lane moves 9 pieces per step
    const uint32_t tq = lane >> 3, tcol = 512u + 8u * (lane & 7u);
    uint32_t i = 0;
    for (uint32_t st = st0; st < steps; st += nwarps, ++i) {
        const uint32_t s = i % S;
        const uint32_t nxt = st + S * nwarps;  // the step that refills stage s
        // its page ids were loaded one step ago; load the following step's now
        const RowLookup look_n = ahead;
        const uint32_t nxt2 = nxt + nwarps;
        ahead = row_lookup(a, s_off, lane < kDynRows && nxt2 < steps ? nxt2 * kDynRows + lane : a.rows);
        if (!mbar_wait(&bars[s], (i / S) & 1u, a.wait_ns)) {
            if (lane == 0) flag(a.err_flags, KVW_ERR_TIMEOUT);
            // leave no copy in flight: wait (bounded) for the stages issued after this one
            for (uint32_t k = 1; k < S && st + k * nwarps < steps; ++k)
                mbar_wait(&bars[(i + k) % S], ((i + k) / S) & 1u, a.wait_ns);
            return;
        }
        const uint32_t valid = (vmask >> (kDynRows * s)) & ((1u << kDynRows) - 1u);
        const unsigned char* sp = stages + (size_t)s * SB;
        // Every row slot of the stage is read and worked on, copied or not (a
        // missing row's codes are never stored), so a step is straight-line
        // code; the rare case (a scale outside div_refined's range) is redone
        // after it.  First pass: the row maxima.
        uint4 raw[kDynRows][2], rtail;
#pragma unroll
        for (uint32_t q = 0; q < kDynRows; ++q) {
            raw[q][0] = staged_raw8<CF8>(sp + q * RB, lane * 8);
            raw[q][1] = staged_raw8<CF8>(sp + q * RB, 256 + lane * 8);
        }
        rtail = staged_raw8<CF8>(sp + tq * RB, tcol);
        const bool vtail = (valid >> tq) & 1u;
        // row maxima as bit patterns of non-negative floats (which order like
        // the values): per lane, then one redux over the warp per row
        uint32_t mq[kDynRows];
        if constexpr (!CF8) {
            const uint32_t atail = halves_max(0u, rtail);
#pragma unroll
            for (uint32_t q = 0; q < kDynRows; ++q) {
                const uint32_t acc = halves_max(halves_max(tq == q ? atail : 0u, raw[q][0]), raw[q][1]);
                const uint32_t m = max(acc & 0x7fffu, (acc >> 16) & 0x7fffu);
                mq[q] = ((valid >> q) & 1u) ? m << 16 : 0u;
            }
        } else {
            const uint32_t mtail = e4m3_piece_max_bits(rtail, a.cache_scale);
#pragma unroll
            for (uint32_t q = 0; q < kDynRows; ++q) {
                const uint32_t m = max(max(e4m3_piece_max_bits(raw[q][0], a.cache_scale),
                                           e4m3_piece_max_bits(raw[q][1], a.cache_scale)),
                                       tq == q ? mtail : 0u);
                mq[q] = ((valid >> q) & 1u) ? m : 0u;
            }
        }
        uint32_t mbits[kDynRows];
#pragma unroll
        for (uint32_t q = 0; q < kDynRows; ++q) mbits[q] = __reduce_max_sync(0xffffffffu, mq[q]);
        // lane q turns row q's maximum into its scale and reciprocal
        uint32_t mine = mbits[0];
#pragma unroll
        for (uint32_t q = 1; q < kDynRows; ++q) mine = lane == q ? mbits[q] : mine;
        const float sc_lane = row_scale(__uint_as_float(mine));
        const float y_lane = __frcp_rn(sc_lane);
        if (lane < kDynRows && ((valid >> lane) & 1u)) scales[(uint64_t)st * kDynRows + lane] = sc_lane;
        float sc[kDynRows], y[kDynRows];
#pragma unroll
        for (uint32_t q = 0; q < kDynRows; ++q) {
            sc[q] = __shfl_sync(0xffffffffu, sc_lane, q);
            y[q] = __shfl_sync(0xffffffffu, y_lane, q);
        }
        float sct = sc[0], yt = y[0];  // the tail piece's row
#pragma unroll
        for (uint32_t q = 1; q < kDynRows; ++q) {
            sct = tq == q ? sc[q] : sct;
            yt = tq == q ? y[q] : yt;
        }
        // Second pass: the pieces read again, a row at a time (the empty asm
        // statements keep the compiler from reusing the first pass's values),
        // and their codes stored where the row was copied (warp-uniform); a
        // row whose scale is outside div_refined's range is stored again
        // below, through the IEEE divide.
        asm volatile("" ::: "memory");
        rtail = staged_raw8<CF8>(sp + tq * RB, tcol);
        unsigned char* const out = a.out + (uint64_t)st * kDynRows * kRow;
        auto put = [&](uint32_t q, uint32_t e, const uint4& v, float scq, float yq, bool fast,
                       bool store) {
            st_if(out + q * kRow + e,
                  CF8 ? quantize_e4m3_piece(v, a.cache_scale, scq, yq, bf16_values && fast)
                      : quantize_bf16_piece(v, scq, yq, fast),
                  store);
        };
#pragma unroll
        for (uint32_t q = 0; q < kDynRows; ++q) {
            asm volatile("" ::: "memory");
            raw[q][0] = staged_raw8<CF8>(sp + q * RB, lane * 8);
            raw[q][1] = staged_raw8<CF8>(sp + q * RB, 256 + lane * 8);
#pragma unroll
            for (uint32_t j = 0; j < 2; ++j)
                put(q, 256u * j + lane * 8, raw[q][j], sc[q], y[q],
                    CF8 ? refined_ok(sc[q]) : true, (valid >> q) & 1u);
        }
        put(tq, tcol, rtail, sct, yt, CF8 ? refined_ok(sct) : true, vtail);
        if constexpr (!CF8) {
            bool slow = vtail && !refined_ok(sct);
#pragma unroll
            for (uint32_t q = 0; q < kDynRows; ++q) slow |= ((valid >> q) & 1u) && !refined_ok(sc[q]);
            if (slow) {
#pragma unroll
                for (uint32_t q = 0; q < kDynRows; ++q)
                    if (((valid >> q) & 1u) && !refined_ok(sc[q]))
#pragma unroll
                        for (uint32_t j = 0; j < 2; ++j)
                            put(q, 256u * j + lane * 8, staged_raw8<CF8>(sp + q * RB, 256u * j + lane * 8),
                                sc[q], y[q], false, true);
                if (vtail && !refined_ok(sct))
                    put(tq, tcol, staged_raw8<CF8>(sp + tq * RB, tcol), sct, yt, false, true);
            }
        }
        // the stage has been read: refill it with step nxt
        fence_proxy_async_smem();
        __syncwarp();
        if (nxt < steps)
            vmask = (vmask & ~(((1u << kDynRows) - 1u) << (kDynRows * s))) |
                    (issue(s, row_resolve(a, look_n)) << (kDynRows * s));
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

template <bool CF8, bool WITHHOLD = false>
cudaError_t launch_dynamic(const GatherArgs& a, float* scales, cudaStream_t stream) {
    constexpr auto k = gather_dynamic_kernel<CF8, WITHHOLD>;
    const size_t smem = dyn_smem<CF8>(a.B);
    uint64_t wave = 0;
    const cudaError_t e = wave_ctas<k>(kDynThreads, smem, wave);
    if (e != cudaSuccess) return e;
    if (wave == 0) return cudaErrorInvalidConfiguration;
    const uint32_t ctas = (a.rows + kDynRows * kDynWarps - 1) / (kDynRows * kDynWarps);
    k<<<ctas < wave ? ctas : (uint32_t)wave, kDynThreads, smem, stream>>>(a, scales);
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
    a.wait_ns = kWaitLimitNs;
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

namespace kvw {
namespace {

int gather_dynamic_entry(void* out_codes, float* out_scales, const kvw_paged_cache_t* cache,
                         uint32_t layer_idx, const uint32_t* ctx_offsets, uint32_t num_batches,
                         uint32_t total_rows, uint32_t* err_flags, cudaStream_t stream,
                         bool withhold, uint64_t wait_ns) {
    if (!cache) return KVW_EINVAL;
    GatherArgs a;
    const int st = make_args(cache, layer_idx, ctx_offsets, num_batches, total_rows, err_flags, a);
    if (st != KVW_OK) return st;
    if (total_rows == 0) return KVW_OK;
    if (!out_codes || !out_scales || !aligned16(out_codes) ||
        (reinterpret_cast<uintptr_t>(out_scales) & 3u) != 0)
        return KVW_EINVAL;
    a.out = static_cast<unsigned char*>(out_codes);
    a.wait_ns = wait_ns;
    const bool cf8 = cache->dtype == KVW_DTYPE_FP8_E4M3;
    cudaError_t e;
#ifdef KVW_TEST_HOOKS
    if (withhold)
        e = cf8 ? launch_dynamic<true, true>(a, out_scales, stream)
                : launch_dynamic<false, true>(a, out_scales, stream);
    else
#else
    if (withhold) return KVW_EUNSUPPORTED;
#endif
        e = cf8 ? launch_dynamic<true>(a, out_scales, stream)
                : launch_dynamic<false>(a, out_scales, stream);
    return e == cudaSuccess ? KVW_OK : KVW_ECUDA;
}

}  // namespace
}  // namespace kvw

extern "C" int kvw_mla_gather_latent_fp8_dynamic(void* out_codes, float* out_scales,
                                                 const kvw_paged_cache_t* cache,
                                                 uint32_t layer_idx, const uint32_t* ctx_offsets,
                                                 uint32_t num_batches, uint32_t total_rows,
                                                 uint32_t* err_flags, cudaStream_t stream) {
    return kvw::gather_dynamic_entry(out_codes, out_scales, cache, layer_idx, ctx_offsets,
                                     num_batches, total_rows, err_flags, stream, false,
                                     kvw::kWaitLimitNs);
}

#ifdef KVW_TEST_HOOKS
// Test builds only (compiled with -DKVW_TEST_HOOKS into a separate library;
// the product library has no such symbol): the dynamic-FP8 gather with the
// first step of every warp announced on its stage barrier but never copied,
// and every wait bounded by `wait_ns`, so each warp's first wait runs out,
// KVW_ERR_TIMEOUT is set and the kernel returns without writing a row.
extern "C" int kvw_test_gather_dynamic_withheld_stage(void* out_codes, float* out_scales,
                                                      const kvw_paged_cache_t* cache,
                                                      uint32_t layer_idx,
                                                      const uint32_t* ctx_offsets,
                                                      uint32_t num_batches, uint32_t total_rows,
                                                      uint32_t* err_flags, cudaStream_t stream,
                                                      uint64_t wait_ns) {
    return kvw::gather_dynamic_entry(out_codes, out_scales, cache, layer_idx, ctx_offsets,
                                     num_batches, total_rows, err_flags, stream, true, wait_ns);
}
#endif
