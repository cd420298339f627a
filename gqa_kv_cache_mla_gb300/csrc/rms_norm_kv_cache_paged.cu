// In-place RMSNorm of the K-cache rows of new tokens.
//
// Operation: "rms_norm_kv_cache_ragged_paged" (Modular MAX kernel API, Mojo
// function page: description of the ragged view built from total_seq_len and
// input_row_offsets, the subset of leading columns given by the length of
// gamma, weight_offset added to gamma, multiply_before_cast; parameter
// per_head_norm).
//
// GB300 design.  A "row" is one (token, kv head) slice of gamma_len leading
// columns (or the whole K row of a token when per_head_norm is off).  A team
// of TL lanes (a power of two, 2..32) owns a row: lane l holds 16-byte
// vectors l, l + TL, ... of it, sums its squares, and an xor-shuffle inside
// the team finishes the reduction, so no shared memory or block barrier is
// needed for the norm itself.  Each team handles RPT rows so every thread has
// RPT x VPL 16-byte loads in flight.  CTAs are persistent (one wave at the
// occupancy the register count allows) and stage the ragged tables and the
// weights once; after that each warp walks its own tiles of teams x RPT rows
// with no block barrier: it resolves the page slots of the few tokens of its
// next tile (ragged lookup in shared memory, page table) into its slice of
// shared memory while the current tile's loads are in flight, then
// normalises the tile and writes it back in place.  Columns at or past
// gamma_len are neither read into the sum nor written.
// Two kernels share this design: rms_norm_rows_kernel, for rows whose
// normalised columns are contiguous and a multiple of 8 wide (per-head
// norms, whole rows of adjacent heads), with the team geometry fixed at
// compile time; and rms_norm_kv_kernel for everything else (ragged gamma
// lengths, whole rows of padded heads), with run-time geometry.
#include <cstdint>

#include "kvw_device.cuh"

namespace kvw {
namespace {

constexpr uint32_t kThreads = 256;
constexpr uint32_t kMaxCols = 2048;
constexpr uint32_t kMaxWarpTileTokens = 66;  // tokens of a warp tile: up to 64 rows + 2

struct KnArgs {
    uint16_t* cache;
    const uint32_t* offsets;
    const uint32_t* cache_lengths;
    const uint32_t* page_table;
    const uint16_t* gamma;
    uint32_t* err_flags;
    int64_t s_page, s_token, s_head, layer_off;
    uint32_t B, T, S, G, max_pages, num_pages, page_size;
    uint32_t rows_per_token;  // num_heads (per-head) or 1 (whole K row)
    uint32_t per_head;
    uint32_t tl_log2;         // team size = 1 << tl_log2
    uint32_t nv;              // 16-byte vectors per row = ceil(G / 8)
    uint32_t rows;            // T * rows_per_token
    float eps, wo;
    float inv_g;              // 1 / gamma_len (rounded)
    uint32_t pt_words;        // page-table words staged in shared memory (0: read from global)
    uint32_t pt_at;           // their word offset in dynamic shared memory
    FastDiv rpt_div;          // division by rows_per_token
    FastDiv ps_div;           // division by page_size
    int mbc;
};

// MBC: multiply_before_cast; FULL: gamma_len is a multiple of 8 (no ragged
// vector).  Both are template parameters so the per-element inner loops are
// branch-free: unpack, square-and-add, scale, weight, pack.
template <int VPL, int RPT, bool MBC, bool FULL>
__global__ void __launch_bounds__(kThreads, 3) rms_norm_kv_kernel(const KnArgs a) {
    extern __shared__ uint32_t s_dyn[];
    uint32_t* s_off = s_dyn;
    uint32_t* s_clen = s_dyn + a.B + 1;
    __shared__ int64_t s_wbase[kThreads / 32][kMaxWarpTileTokens];

    const uint32_t TL = 1u << a.tl_log2;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t team = lane >> a.tl_log2;   // team inside the warp
    const uint32_t tl = lane & (TL - 1u);
    const uint32_t teams = 32u >> a.tl_log2;   // teams per warp

    // weights gamma + weight_offset of the normalised columns, in shared memory
    // (zero past gamma_len), read as float4 pairs by the lanes of each column
    __shared__ __align__(16) float s_w[kMaxCols];
    const uint32_t gcols = a.nv * 8u;
    for (uint32_t c = threadIdx.x; c < gcols; c += kThreads)
        s_w[c] = c < a.G ? __fadd_rn(bf16_lo(__ldg(a.gamma + c)), a.wo) : 0.0f;

    if (!stage_ragged(a.offsets, a.cache_lengths, a.B, a.T, s_off, s_clen)) {
        if (threadIdx.x == 0) flag(a.err_flags, KVW_ERR_OFFSETS);
        return;
    }
    // Warp tiles of teams x RPT consecutive rows, walked by each warp on its
    // own (no block barrier after the set-up above).  The page slot of every
    // token of a tile sits in the warp's slice of shared memory: the warp
    // resolves the next tile's slots after reading the current ones and
    // while the current tile's loads are in flight.
    const uint32_t rows_wt = teams * RPT;
    const uint32_t wtiles = (a.rows + rows_wt - 1) / rows_wt;
    const uint32_t nwarps = gridDim.x * (kThreads / 32);
    int64_t* wbase = s_wbase[warp];
    auto resolve = [&](uint32_t wt) {
        const uint32_t r0 = wt * rows_wt;
        const uint32_t t_lo = fast_div(r0, a.rpt_div);
        const uint32_t t_hi = fast_div(min(r0 + rows_wt, a.rows) - 1, a.rpt_div);
        for (uint32_t k = lane; k <= t_hi - t_lo; k += 32) {
            const uint32_t t = t_lo + k;
            const uint32_t b = find_request(s_off, a.B, t);
            const uint64_t pos = (uint64_t)s_clen[b] + (t - s_off[b]);
            const int64_t base = slot_row(a.page_table, a.max_pages, a.num_pages, a.ps_div,
                                          a.s_page, a.s_token, a.layer_off, b, pos);
            wbase[k] = base;
            if (base < 0) flag(a.err_flags, KVW_ERR_PAGE);
        }
    };
    uint32_t wt = blockIdx.x * (kThreads / 32) + warp;
    if (wt < wtiles) resolve(wt);
    __syncwarp();

    for (; wt < wtiles; wt += nwarps) {
    const uint32_t r0 = wt * rows_wt;
    const uint32_t t_lo = fast_div(r0, a.rpt_div);
    const uint32_t r_end = min(r0 + rows_wt, a.rows);

    // pointers of this lane's first vector in each of its rows (null: no row);
    // row r = r0 + team + q * teams, walked as (token, head) without dividing
    uint16_t* ptr[RPT];
    uint4 x[RPT][VPL];
    uint32_t t = fast_div(r0 + team, a.rpt_div);
    uint32_t g = (r0 + team) - t * a.rows_per_token;
    const uint32_t dt = fast_div(teams, a.rpt_div), dg = teams - dt * a.rows_per_token;
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
        const uint32_t r = r0 + team + q * teams;
        ptr[q] = nullptr;
        if (r < r_end) {
            const int64_t base = wbase[t - t_lo];
            if (base >= 0) ptr[q] = a.cache + base + (a.per_head ? (int64_t)g * a.s_head : 0);
        }
        t += dt;
        g += dg;
        if (g >= a.rows_per_token) {
            g -= a.rows_per_token;
            ++t;
        }
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            x[q][v] = make_uint4(0, 0, 0, 0);
            const uint32_t c = (tl + v * TL) * 8u;  // column inside the normalised row
            if (ptr[q] && c < a.G) {
                const uint32_t off = a.per_head ? c : (c / a.S) * (uint32_t)a.s_head + (c % a.S);
                x[q][v] = *reinterpret_cast<const uint4*>(ptr[q] + off);
            }
        }
    }
    __syncwarp();  // every lane has read this tile's slots
    if (wt + nwarps < wtiles) resolve(wt + nwarps);
    __syncwarp();  // the next tile's slots are visible to the whole warp

#pragma unroll
    for (int q = 0; q < RPT; ++q) {
        float xs[VPL][8];
        float ss = 0.0f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            unpack8(x[q][v], xs[v]);
            const uint32_t c = (tl + v * TL) * 8u;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (FULL || c + e < a.G) ss = __fadd_rn(ss, __fmul_rn(xs[v][e], xs[v][e]));
        }
        for (uint32_t o = TL >> 1; o > 0; o >>= 1)
            ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        if (!ptr[q]) continue;
        const float rinv = rms_inv(ss, (float)a.G, a.eps);
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            const uint32_t c = (tl + v * TL) * 8u;
            if (c >= a.G) continue;
            const float4 w0 = *reinterpret_cast<const float4*>(s_w + c);
            const float4 w1 = *reinterpret_cast<const float4*>(s_w + c + 4);
            const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float xr = __fmul_rn(xs[v][e], rinv);
                y[e] = MBC ? __fmul_rn(xr, w[e])
                           : __fmul_rn(__bfloat162float(__float2bfloat16_rn(xr)), w[e]);
            }
            const uint4 out = pack8_bf16(y);
            uint16_t* dst =
                ptr[q] + (a.per_head ? c : (c / a.S) * (uint32_t)a.s_head + (c % a.S));
            if (FULL || c + 8u <= a.G) {
                *reinterpret_cast<uint4*>(dst) = out;
            } else {  // ragged tail of the gamma-length slice: columns < G only
                const uint32_t words[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (c + e < a.G) dst[e] = (uint16_t)(e & 1 ? words[e >> 1] >> 16 : words[e >> 1]);
            }
        }
    }
    }
}

// Exact bf16 widening by byte permutes: the same values as unpack8, from a
// different instruction sequence.  The sum-of-squares pass uses this one and
// the output pass unpack8, so the compiler re-widens the packed rows for the
// output pass instead of keeping every widened value of the tile live across
// the team reduction.
__device__ __forceinline__ void unpack8_perm(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(__byte_perm(w[i], 0u, 0x1044u));
        f[2 * i + 1] = __uint_as_float(__byte_perm(w[i], 0u, 0x3244u));
    }
}

// Fast path for contiguous rows: the normalised columns of a row are adjacent
// in memory (per-head norm, or the whole K row of a token whose heads are
// adjacent) and gamma_len is a multiple of 8.  The team geometry (TL lanes,
// VPL 16-byte vectors per lane, RPT rows per team) is compile-time, so lane
// tl of a team owns columns 8 (tl + v TL) .. + 7 of every row of the launch:
// a row is one base pointer plus constant offsets and the team reduction
// unrolls.  The sum of squares runs as VPL independent fused multiply-add
// chains; team lane q computes the 1/rms of row q of its team (rsqrt refined
// by one Newton-Raphson step, r' = r (3 - m r^2) / 2, within two fp32 ulp of
// the correctly rounded value, so a bf16 result differs from a correctly
// rounded reference by at most one ulp, on a few elements in 10^5) and the
// team reads the values back with shuffles.  Slot resolution, tiling and the
// per-warp walk are those of rms_norm_kv_kernel; a small page table can be
// staged in shared memory with the ragged tables (see launch_rows).
template <int TL, int VPL, int RPT, bool MBC>
__global__ void __launch_bounds__(kThreads, 4) rms_norm_rows_kernel(const KnArgs a) {
    static_assert(RPT <= TL, "a team lane computes the 1/rms of one row of its team");
    constexpr uint32_t kTeams = 32u / TL;
    constexpr uint32_t kRowsWt = kTeams * RPT;  // rows of a warp tile
    constexpr uint32_t kCols = TL * VPL * 8;     // columns a team covers
    extern __shared__ uint32_t s_dyn[];
    uint32_t* s_off = s_dyn;
    uint32_t* s_clen = s_dyn + a.B + 1;
    uint32_t* s_pt = s_dyn + a.pt_at;
    __shared__ int64_t s_wbase[kThreads / 32][kRowsWt + 2];
    __shared__ __align__(16) float s_w[kCols];

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t team = lane / TL, tl = lane % TL;
    // a small page table is copied to shared memory with the ragged tables
    // (asynchronous 4-byte copies, complete before the staging barrier) when
    // warps walk several tiles, so that resolving the slots of a tile needs no
    // further global round trip
    for (uint32_t i = threadIdx.x; i < a.pt_words; i += kThreads)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(s_pt + i)),
                     "l"(a.page_table + i)
                     : "memory");
    // weights gamma + weight_offset of the normalised columns (zero past
    // gamma_len, whose vectors are never loaded, normalised or stored)
    for (uint32_t c = threadIdx.x; c < kCols; c += kThreads)
        s_w[c] = c < a.G ? __fadd_rn(bf16_lo(__ldg(a.gamma + c)), a.wo) : 0.0f;
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (!stage_ragged(a.offsets, a.cache_lengths, a.B, a.T, s_off, s_clen)) {
        if (threadIdx.x == 0) flag(a.err_flags, KVW_ERR_OFFSETS);
        return;
    }
    const uint32_t wtiles = (a.rows + kRowsWt - 1) / kRowsWt;
    const uint32_t nwarps = gridDim.x * (kThreads / 32);
    int64_t* wbase = s_wbase[warp];
    // divisions by rows_per_token and page_size are multiply-highs (FastDiv)
    auto resolve = [&](uint32_t wt) {
        const uint32_t r0 = wt * kRowsWt;
        const uint32_t t_lo = fast_div(r0, a.rpt_div);
        const uint32_t t_hi = fast_div(min(r0 + kRowsWt, a.rows) - 1, a.rpt_div);
        for (uint32_t k = lane; k <= t_hi - t_lo; k += 32) {
            const uint32_t t = t_lo + k;
            const uint32_t b = find_request(s_off, a.B, t);
            const uint64_t pos = (uint64_t)s_clen[b] + (t - s_off[b]);
            int64_t base = -1;
            if ((pos >> 32) == 0) {  // no page table reaches past 32-bit positions
                const uint32_t p32 = (uint32_t)pos;
                const uint32_t pidx = fast_div(p32, a.ps_div);
                if (pidx < a.max_pages) {
                    const uint32_t page = a.pt_words ? s_pt[b * a.max_pages + pidx]
                                                     : __ldg(a.page_table + (uint64_t)b * a.max_pages + pidx);
                    if (page < a.num_pages)
                        base = (int64_t)page * a.s_page + a.layer_off +
                               (int64_t)(p32 - pidx * a.page_size) * a.s_token;
                }
            }
            wbase[k] = base;
            if (base < 0) flag(a.err_flags, KVW_ERR_PAGE);
        }
    };
    uint32_t wt = blockIdx.x * (kThreads / 32) + warp;
    if (wt < wtiles) resolve(wt);
    __syncwarp();

    const uint32_t nvec = a.nv;
    for (; wt < wtiles; wt += nwarps) {
        const uint32_t r0 = wt * kRowsWt;
        const uint32_t t_lo = fast_div(r0, a.rpt_div);
        const uint32_t r_end = min(r0 + kRowsWt, a.rows);
        // row r = r0 + team + q * kTeams, walked as (token, head) without dividing
        uint16_t* ptr[RPT];
        uint4 x[RPT][VPL];
        uint32_t t = fast_div(r0 + team, a.rpt_div);
        uint32_t g = (r0 + team) - t * a.rows_per_token;
        const uint32_t dt = fast_div(kTeams, a.rpt_div), dg = kTeams - dt * a.rows_per_token;
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            const uint32_t r = r0 + team + q * kTeams;
            ptr[q] = nullptr;
            if (r < r_end) {
                const int64_t base = wbase[t - t_lo];
                if (base >= 0) ptr[q] = a.cache + base + (int64_t)g * a.s_head + tl * 8u;
            }
            t += dt;
            g += dg;
            if (g >= a.rows_per_token) {
                g -= a.rows_per_token;
                ++t;
            }
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                x[q][v] = make_uint4(0, 0, 0, 0);
                if (ptr[q] && tl + v * TL < nvec)
                    x[q][v] = *reinterpret_cast<const uint4*>(ptr[q] + v * TL * 8);
            }
        }
        __syncwarp();  // every lane has read this tile's slots
        if (wt + nwarps < wtiles) resolve(wt + nwarps);
        __syncwarp();  // the next tile's slots are visible to the whole warp

        // sums of squares of the RPT rows, completed across the team
        float ss[RPT];
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            float part[VPL];
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                float xs[8];
                unpack8_perm(x[q][v], xs);
                part[v] = __fmul_rn(xs[0], xs[0]);
#pragma unroll
                for (int e = 1; e < 8; ++e) part[v] = __fmaf_rn(xs[e], xs[e], part[v]);
            }
#pragma unroll
            for (int v = 1; v < VPL; ++v) part[0] = __fadd_rn(part[0], part[v]);
            ss[q] = part[0];
#pragma unroll
            for (int o = TL / 2; o > 0; o >>= 1)
                ss[q] = __fadd_rn(ss[q], __shfl_xor_sync(0xffffffffu, ss[q], o));
        }
        // one 1/rms per row: team lane q computes row q's
        // and the team reads them back, instead of every lane computing all
        float mine = ss[0];
#pragma unroll
        for (int q = 1; q < RPT; ++q)
            if (tl == (uint32_t)q) mine = ss[q];
        const float m = __fadd_rn(__fmul_rn(mine, a.inv_g), a.eps);
        const float est = rsqrtf(m);
        const float rinv_mine = __fmul_rn(est, __fmaf_rn(__fmul_rn(-0.5f, m) * est, est, 1.5f));
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            const float rinv = __shfl_sync(0xffffffffu, rinv_mine, (lane & ~(TL - 1u)) | q);
            if (!ptr[q]) continue;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                if (tl + v * TL >= nvec) continue;
                const float4 w0 = *reinterpret_cast<const float4*>(s_w + (tl + v * TL) * 8u);
                const float4 w1 = *reinterpret_cast<const float4*>(s_w + (tl + v * TL) * 8u + 4);
                const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                float xs[8], y[8];
                unpack8(x[q][v], xs);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float xr = __fmul_rn(xs[e], rinv);
                    y[e] = MBC ? __fmul_rn(xr, wv[e])
                               : __fmul_rn(__bfloat162float(__float2bfloat16_rn(xr)), wv[e]);
                }
                *reinterpret_cast<uint4*>(ptr[q] + v * TL * 8) = pack8_bf16(y);
            }
        }
    }
}

// `smem` holds the ragged tables; `pt_words` page-table words may be staged
// behind them (at word a.pt_at).  Staging costs every CTA the copy of the
// whole table before its first slot resolution and saves a global round trip
// on each later one, so it is used when warps walk 1.5 or more tiles on
// average (same-box A/B: 9% faster with 1.7-2.3 tiles per warp, 3% slower
// with 1.1).
template <int TL, int VPL, int RPT, bool MBC>
cudaError_t launch_rows(const KnArgs& a, size_t smem, uint32_t pt_words, cudaStream_t stream) {
    constexpr auto k = rms_norm_rows_kernel<TL, VPL, RPT, MBC>;
    constexpr uint32_t rows_wt = (32u / TL) * RPT;
    const uint32_t wtiles = (a.rows + rows_wt - 1) / rows_wt;
    const uint32_t tiles = (wtiles + kThreads / 32 - 1) / (kThreads / 32);  // CTAs with work
    const size_t smem_pt = sizeof(uint32_t) * ((size_t)a.pt_at + pt_words);
    uint64_t wave = 0;
    cudaError_t e = wave_ctas<k>(kThreads, pt_words ? smem_pt : smem, wave);
    if (e != cudaSuccess) return e;
    if (wave == 0) return cudaErrorInvalidConfiguration;
    const uint32_t grid = tiles < wave ? tiles : (uint32_t)wave;
    KnArgs b = a;
    b.pt_words = 2ull * wtiles >= 3ull * grid * (kThreads / 32) ? pt_words : 0u;
    k<<<grid, kThreads, b.pt_words ? smem_pt : smem, stream>>>(b);
    return cudaGetLastError();
}

// Team geometry of the contiguous-row path from the 16-byte vectors per row
// (nv <= 128): narrow teams for short rows, so that one instruction stream
// serves several rows and every lane keeps a few vectors in flight.
template <bool MBC>
cudaError_t launch_rows_for(const KnArgs& a, size_t smem, uint32_t pt_words, cudaStream_t stream) {
    if (a.nv <= 4) return launch_rows<4, 1, 4, MBC>(a, smem, pt_words, stream);
    if (a.nv <= 8) return launch_rows<4, 2, 4, MBC>(a, smem, pt_words, stream);
    if (a.nv <= 16) return launch_rows<4, 4, 2, MBC>(a, smem, pt_words, stream);
    if (a.nv <= 32) return launch_rows<8, 4, 2, MBC>(a, smem, pt_words, stream);
    if (a.nv <= 64) return launch_rows<16, 4, 2, MBC>(a, smem, pt_words, stream);
    // whole K rows (up to 1024 columns): two rows per team measured 11% faster than one
    return launch_rows<32, 4, 2, MBC>(a, smem, pt_words, stream);
}

template <int VPL, int RPT, bool MBC, bool FULL>
cudaError_t launch_one(const KnArgs& a, size_t smem, cudaStream_t stream) {
    constexpr auto k = rms_norm_kv_kernel<VPL, RPT, MBC, FULL>;
    const uint32_t rows_wt = (32u >> a.tl_log2) * RPT;
    const uint32_t wtiles = (a.rows + rows_wt - 1) / rows_wt;
    const uint32_t tiles = (wtiles + kThreads / 32 - 1) / (kThreads / 32);  // CTAs with work
    uint64_t wave = 0;
    const cudaError_t e = wave_ctas<k>(kThreads, smem, wave);
    if (e != cudaSuccess) return e;
    if (wave == 0) return cudaErrorInvalidConfiguration;
    k<<<tiles < wave ? tiles : (uint32_t)wave, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int VPL, int RPT>
cudaError_t launch(const KnArgs& a, size_t smem, cudaStream_t stream) {
    const bool full = a.G % 8 == 0;
    if (a.mbc)
        return full ? launch_one<VPL, RPT, true, true>(a, smem, stream)
                    : launch_one<VPL, RPT, true, false>(a, smem, stream);
    return full ? launch_one<VPL, RPT, false, true>(a, smem, stream)
                : launch_one<VPL, RPT, false, false>(a, smem, stream);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvw

extern "C" int kvw_rms_norm_kv_cache_paged(const kvw_paged_cache_t* cache, const void* gamma,
                                           uint32_t gamma_len, float epsilon, float weight_offset,
                                           uint32_t layer_idx, uint32_t total_seq_len,
                                           const uint32_t* input_row_offsets, uint32_t num_batches,
                                           int multiply_before_cast, int per_head_norm,
                                           uint32_t* err_flags, cudaStream_t stream) {
    using namespace kvw;
    if (!cache) return KVW_EINVAL;
    if (cache->dtype != KVW_DTYPE_BF16) return KVW_EUNSUPPORTED;
    const uint32_t S = cache->head_size;
    if (S == 0 || S % 8 != 0) return KVW_EINVAL;
    if (num_batches > KVW_MAX_BATCHES) return KVW_EUNSUPPORTED;
    if (gamma_len == 0) return KVW_EINVAL;
    if (per_head_norm ? gamma_len > S : (uint64_t)gamma_len != (uint64_t)S * cache->num_heads)
        return KVW_EINVAL;
    if (gamma_len > kMaxCols) return KVW_EUNSUPPORTED;
    if (total_seq_len == 0 || cache->num_heads == 0) return KVW_OK;
    if (!gamma || !input_row_offsets || !cache->data || !cache->page_table || !cache->cache_lengths)
        return KVW_EINVAL;
    if (layer_idx >= cache->num_layers || cache->page_size == 0 || cache->max_pages_per_seq == 0)
        return KVW_EINVAL;
    if (!(epsilon >= 0.0f)) return KVW_EINVAL;
    if (!aligned16(gamma) || !aligned16(cache->data)) return KVW_EINVAL;
    if ((cache->stride_page * 2) % 16 || (cache->stride_layer * 2) % 16 ||
        (cache->stride_token * 2) % 16 || (cache->stride_head * 2) % 16 ||
        cache->stride_page <= 0 || cache->stride_token <= 0)
        return KVW_EINVAL;

    KnArgs a;
    a.cache = static_cast<uint16_t*>(cache->data);
    a.offsets = input_row_offsets;
    a.cache_lengths = cache->cache_lengths;
    a.page_table = cache->page_table;
    a.gamma = static_cast<const uint16_t*>(gamma);
    a.err_flags = err_flags;
    a.s_page = cache->stride_page;
    a.s_token = cache->stride_token;
    a.s_head = cache->stride_head;
    a.layer_off = (int64_t)layer_idx * cache->stride_layer;
    a.B = num_batches;
    a.T = total_seq_len;
    a.S = S;
    a.G = gamma_len;
    a.max_pages = cache->max_pages_per_seq;
    a.num_pages = cache->num_pages;
    a.page_size = cache->page_size;
    a.per_head = per_head_norm ? 1u : 0u;
    a.rows_per_token = per_head_norm ? cache->num_heads : 1u;
    a.rpt_div = make_fast_div(a.rows_per_token);
    a.ps_div = make_fast_div(cache->page_size);
    a.nv = (gamma_len + 7) / 8;
    // Team of TL lanes per row, each lane VPL 16-byte vectors: narrow teams
    // (4 lanes for up to 16 vectors) let one instruction stream serve many
    // rows, so the per-row work (shuffles, the reciprocal square root,
    // addressing) is shared by more rows per warp.
    uint32_t tl = 4;
    while (tl < 32 && tl * 4 < a.nv) tl <<= 1;
    a.tl_log2 = 0;
    while ((1u << a.tl_log2) < tl) ++a.tl_log2;
    const uint32_t vpl = (a.nv + tl - 1) / tl;
    const uint64_t rows = (uint64_t)total_seq_len * a.rows_per_token;
    if (rows > 0xfffff000ull) return KVW_EUNSUPPORTED;
    a.rows = (uint32_t)rows;
    a.eps = epsilon;
    a.wo = weight_offset;
    a.inv_g = 1.0f / (float)gamma_len;
    a.mbc = multiply_before_cast ? 1 : 0;
    // page tables up to 16 KiB may be staged in shared memory by the contiguous-row kernel
    const uint64_t pt_all = (uint64_t)num_batches * cache->max_pages_per_seq;
    const uint32_t pt_words = pt_all * 4 <= 16384 ? (uint32_t)pt_all : 0u;
    a.pt_words = 0;
    a.pt_at = 2 * num_batches + 1;
    const size_t smem = sizeof(uint32_t) * (2 * (size_t)num_batches + 1);
    cudaError_t e;
    // contiguous rows of whole vectors take the fast path; gamma lengths that
    // are not a multiple of 8 and whole K rows of padded heads the general one
    const bool contiguous = per_head_norm || cache->num_heads == 1 ||
                            cache->stride_head == (int64_t)S;
    if (contiguous && gamma_len % 8 == 0 && a.nv <= 128)
        e = a.mbc ? launch_rows_for<true>(a, smem, pt_words, stream)
                  : launch_rows_for<false>(a, smem, pt_words, stream);
    else if (vpl <= 1)
        e = launch<1, 8>(a, smem, stream);
    else if (vpl <= 2)
        e = launch<2, 4>(a, smem, stream);
    else if (vpl <= 4)
        e = launch<4, 2>(a, smem, stream);
    else
        e = launch<8, 1>(a, smem, stream);
    return e == cudaSuccess ? KVW_OK : KVW_ECUDA;
}
