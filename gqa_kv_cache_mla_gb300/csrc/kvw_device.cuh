// Device helpers shared by the three KV-cache write kernels (sm_103a).
//
// Everything here is memory plumbing and exact arithmetic building blocks:
// 16-byte vector loads/stores with cache hints, exact bf16 widening, packed
// bf16 / FP8 E4M3 conversion through the hardware cvt instructions, the
// rotation of one pair, and the per-CTA ragged lookup (input_row_offsets ->
// request -> slot position) that every kernel starts with.
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kvw.h"

namespace kvw {

// ------------------------------------------------------------ memory access

// Read-once stream (activations): evict-first in L1 and L2.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
// Write-once stream (outputs nobody rereads in this kernel).
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }
// Small tables reused by many CTAs (gamma, freqs rows, offsets): read-only path.
__device__ __forceinline__ uint4 ld_table(const uint4* p) { return __ldg(p); }
__device__ __forceinline__ float4 ld_table(const float4* p) { return __ldg(p); }

// ------------------------------------------------------------ conversions

// bf16 -> fp32 is exact: the bf16 pattern is the upper half of the fp32 one.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Two fp32 -> packed bf16x2, round to nearest even (one cvt.rn.bf16x2.f32).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8_bf16(const float (&f)[8]) {
    uint4 v;
    v.x = pack_bf16x2(f[0], f[1]);
    v.y = pack_bf16x2(f[2], f[3]);
    v.z = pack_bf16x2(f[4], f[5]);
    v.w = pack_bf16x2(f[6], f[7]);
    return v;
}

// Two fp32 -> packed E4M3x2, round to nearest even, saturating to +-448
// (one cvt.rn.satfinite.e4m3x2.f32).  Element `lo` lands in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint2 pack8_e4m3(const float (&f)[8]) {
    uint2 v;
    v.x = pack_e4m3x2(f[0], f[1]) | (pack_e4m3x2(f[2], f[3]) << 16);
    v.y = pack_e4m3x2(f[4], f[5]) | (pack_e4m3x2(f[6], f[7]) << 16);
    return v;
}

// Eight E4M3 codes (little-endian in a uint2) -> fp32, exact (E4M3 values
// are a subset of fp16, converted with cvt.f16x2.e4m3x2).
__device__ __forceinline__ void unpack8_e4m3(const uint2& v, float (&f)[8]) {
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_fp8x2_storage_t pair =
            static_cast<__nv_fp8x2_storage_t>((w[i >> 1] >> (16 * (i & 1))) & 0xffffu);
        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
        const float2 x = __half22float2(__half2(h));
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}

// Eight key-cache elements at byte address p as fp32: bf16 widened exactly,
// or E4M3 decoded and multiplied by the per-tensor scale.
template <bool FP8>
__device__ __forceinline__ void load_k8(const unsigned char* p, float (&f)[8], float scale) {
    if constexpr (FP8) {
        unpack8_e4m3(*reinterpret_cast<const uint2*>(p), f);
        if (scale != 1.0f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], scale);
        }
    } else {
        unpack8(*reinterpret_cast<const uint4*>(p), f);
    }
}

// Eight fp32 values stored as key-cache elements: bf16 round to nearest
// even, or E4M3 satfinite(y / scale).
template <bool FP8>
__device__ __forceinline__ void store_k8(unsigned char* p, const float (&y)[8], float scale) {
    if constexpr (FP8) {
        float z[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) z[i] = scale == 1.0f ? y[i] : __fdiv_rn(y[i], scale);
        *reinterpret_cast<uint2*>(p) = pack8_e4m3(z);
    } else {
        *reinterpret_cast<uint4*>(p) = pack8_bf16(y);
    }
}

// ------------------------------------------------------------ arithmetic

// Rotation of one pair by (c, s) = (cos, sin): y0 = x0*c - x1*s,
// y1 = x0*s + x1*c.  The _rn intrinsics keep every product rounded on its
// own (never contracted into an FMA), so the result is the IEEE fp32 value
// of that expression evaluated term by term.
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float& y0,
                                          float& y1) {
    y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    y1 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
}

// 1 / sqrt(ss / n + eps) with correctly rounded divide and square root.
__device__ __forceinline__ float rms_inv(float ss, float n, float eps) {
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, n), eps)));
}

// x / s for the dynamic FP8 quantisers, from y = RN(1/s) and one FMA
// correction step (Markstein's division refinement: P. Markstein, IBM J. Res.
// Dev. 34(1), 1990): q0 = RN(x*y), r = x - q0*s (exact with an FMA),
// q = RN(q0 + r*y), the correctly rounded quotient while s, 1/s and the
// remainder are normal.  Used for scales in [2^-60, 2^60] (refined_ok) on
// bf16 values x with s = RN(amax / 448), amax a bf16 magnitude, where every
// quotient of magnitude >= 2^-14 keeps all three normal and smaller ones give
// an E4M3 zero whatever their last bits; copysignf keeps the sign of x on a
// zero result.
__device__ __forceinline__ float div_refined(float x, float s, float y) {
    const float q0 = __fmul_rn(x, y);
    const float r = __fmaf_rn(-q0, s, x);
    return copysignf(__fmaf_rn(r, y, q0), x);
}

__device__ __forceinline__ bool refined_ok(float sc) { return sc >= 0x1p-60f && sc <= 0x1p60f; }

__device__ __forceinline__ void flag(uint32_t* err_flags, uint32_t bits) {
    if (err_flags) atomicOr(err_flags, bits);
}

// Unsigned 32-bit division by a run-time invariant d >= 1 as a multiply-high,
// an add and a shift (T. Granlund and P. L. Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, section 4): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1 (m < 2^32),
// floor(n / d) = (umulhi(m, n) + n) >> l for every 32-bit n, the sum taken
// in 64 bits.  The host computes (m, l) once per launch (make_fast_div).
struct FastDiv {
    uint32_t d, m, l;
};

inline FastDiv make_fast_div(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.l = 0;
    while ((1ull << f.l) < d) ++f.l;
    f.m = (uint32_t)(((((uint64_t)1 << f.l) - d) << 32) / d + 1);
    return f;
}

__host__ __device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
    const uint32_t hi = __umulhi(f.m, n);
#else
    const uint32_t hi = (uint32_t)(((uint64_t)f.m * n) >> 32);
#endif
    return (uint32_t)(((uint64_t)hi + n) >> f.l);
}

// ------------------------------------------------------------ ragged lookup

// Ragged metadata staging for the pipelined kernels (GQA, K norm): each
// thread loads its slices of offsets[i], offsets[i+1] and cache_lengths[i]
// into registers (issue), then writes the shared copy, checks that the
// offsets start at 0, never decrease and end at T, and returns that verdict
// through one barrier (commit).  Every thread of the CTA must call both; the
// verdict is uniform.
struct RaggedLoads {
    static constexpr int kRegRounds = 2;
    uint32_t off[kRegRounds], nxt[kRegRounds], clen[kRegRounds];

    __device__ __forceinline__ void issue(const uint32_t* __restrict__ offsets,
                                          const uint32_t* __restrict__ cache_lengths,
                                          uint32_t B) {
#pragma unroll
        for (int k = 0; k < kRegRounds; ++k) {
            const uint32_t i = threadIdx.x + k * blockDim.x;
            off[k] = nxt[k] = clen[k] = 0;
            if (i <= B) off[k] = __ldg(offsets + i);
            if (i < B) {
                nxt[k] = __ldg(offsets + i + 1);
                clen[k] = __ldg(cache_lengths + i);
            }
        }
    }

    __device__ __forceinline__ bool commit(const uint32_t* __restrict__ offsets,
                                           const uint32_t* __restrict__ cache_lengths,
                                           uint32_t B, uint32_t T, uint32_t* s_off,
                                           uint32_t* s_clen) const {
        int ok = 1;
#pragma unroll
        for (int k = 0; k < kRegRounds; ++k) {
            const uint32_t i = threadIdx.x + k * blockDim.x;
            if (i <= B) {
                s_off[i] = off[k];
                if ((i == 0 && off[k] != 0u) || (i == B && off[k] != T)) ok = 0;
            }
            if (i < B) {
                s_clen[i] = clen[k];
                if (off[k] > nxt[k]) ok = 0;
            }
        }
        for (uint32_t i = threadIdx.x + kRegRounds * blockDim.x; i <= B; i += blockDim.x) {
            const uint32_t o = __ldg(offsets + i);
            s_off[i] = o;
            if (i < B) {
                s_clen[i] = __ldg(cache_lengths + i);
                if (o > __ldg(offsets + i + 1)) ok = 0;
            }
            if (i == B && o != T) ok = 0;
        }
        return __syncthreads_and(ok) != 0;
    }
};

// Both halves at once.
__device__ __forceinline__ bool stage_ragged(const uint32_t* __restrict__ offsets,
                                             const uint32_t* __restrict__ cache_lengths,
                                             uint32_t B, uint32_t T, uint32_t* s_off,
                                             uint32_t* s_clen) {
    RaggedLoads r;
    r.issue(offsets, cache_lengths, B);
    return r.commit(offsets, cache_lengths, B, T, s_off, s_clen);
}

// Request owning token t, for validated offsets (offsets[0] = 0 <= t <
// offsets[B] = T): the largest b with offsets[b] <= t.  Binary search over
// the staged copy.
__device__ __forceinline__ uint32_t find_request(const uint32_t* s_off, uint32_t B, uint32_t t) {
    uint32_t lo = 0, hi = B;  // s_off[lo] <= t < s_off[hi]
    while (hi - lo > 1u) {
        uint32_t mid = (lo + hi) >> 1;
        if (s_off[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Page id of slot `pos` of request b, or KVW_PAGE_UNMAPPED when the page
// index is past the table (callers compare the result with num_pages).
__device__ __forceinline__ uint32_t page_of(const uint32_t* __restrict__ page_table,
                                           uint32_t max_pages, uint32_t page_size, uint32_t b,
                                           uint64_t pos) {
    const uint64_t pidx = pos / page_size;
    return pidx < max_pages ? __ldg(page_table + (uint64_t)b * max_pages + pidx)
                            : KVW_PAGE_UNMAPPED;
}

// Element offset of the K row of slot `pos` of request b in `layer_off`, or
// -1 when the slot maps to no valid page.  `ps` divides by the page size.
__device__ __forceinline__ int64_t slot_row(const uint32_t* __restrict__ page_table,
                                           uint32_t max_pages, uint32_t num_pages,
                                           const FastDiv& ps, int64_t s_page, int64_t s_token,
                                           int64_t layer_off, uint32_t b, uint64_t pos) {
    if (pos >> 32) return -1;  // no page table reaches that far (max_pages is 32-bit)
    const uint32_t p32 = (uint32_t)pos;
    const uint32_t pidx = fast_div(p32, ps), row = p32 - pidx * ps.d;
    if (pidx >= max_pages) return -1;
    const uint32_t page = __ldg(page_table + (uint64_t)b * max_pages + pidx);
    if (page >= num_pages) return -1;
    return (int64_t)page * s_page + layer_off + (int64_t)row * s_token;
}

// ------------------------------------------------------------ TMA + mbarrier

// Shared-memory address of a generic pointer into shared memory.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of parity `parity` to complete, giving up after
// `limit_ns` nanoseconds (returns false then).  No wait in this library is
// unbounded.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// One bulk (TMA) copy global -> shared, completing on `bar` with `bytes`
// transaction bytes.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// ------------------------------------------------------------ host: launch facts

// The launchers run on every call of a serving loop, where a driver query per
// call would cost about as much as a decode kernel.  The facts below are
// queried once per device (occupancy once per kernel instance, device and
// launch shape) and kept for the life of the process; the cached words are
// read and written atomically, so concurrent callers at worst repeat a query.
constexpr int kMaxDevices = 64;

// Attribute ATTR of the current device.
template <int ATTR>
inline cudaError_t device_attr(int& out) {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (cacheable) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) {
            out = v;
            return cudaSuccess;
        }
    }
    e = cudaDeviceGetAttribute(&out, static_cast<cudaDeviceAttr>(ATTR), dev);
    if (e == cudaSuccess && cacheable && out > 0) cache[dev].store(out, std::memory_order_relaxed);
    return e;
}

inline cudaError_t sm_count(int& out) { return device_attr<cudaDevAttrMultiProcessorCount>(out); }
inline cudaError_t smem_optin(int& out) {
    return device_attr<cudaDevAttrMaxSharedMemoryPerBlockOptin>(out);
}

// Allow kernel K `smem` bytes of dynamic shared memory on the current device
// (the attribute is raised once per device to the largest size asked for).
template <auto K>
inline cudaError_t prepare_smem(size_t smem) {
    static std::atomic<uint64_t> allowed[kMaxDevices];
    if (smem == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (cacheable && allowed[dev].load(std::memory_order_relaxed) >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess || !cacheable) return e;
    uint64_t prev = allowed[dev].load(std::memory_order_relaxed);
    while (prev < smem && !allowed[dev].compare_exchange_weak(prev, smem)) {
    }
    return cudaSuccess;
}

// CTAs of kernel K resident on the whole current device at once with
// `threads` threads and `smem` bytes of dynamic shared memory (0 when none
// fits); also allows K that much shared memory.
template <auto K>
inline cudaError_t wave_ctas(int threads, size_t smem, uint64_t& out) {
    static std::atomic<uint64_t> occ[kMaxDevices];  // smem << 24 | threads << 8 | per SM
    cudaError_t e = prepare_smem<K>(smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = sm_count(sms)) != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    const uint64_t key = ((uint64_t)smem << 24) | ((uint64_t)threads << 8);
    if (cacheable) {
        const uint64_t v = occ[dev].load(std::memory_order_relaxed);
        if ((v & ~0xffull) == key && (v & 0xffull) != 0) {
            out = (uint64_t)sms * (v & 0xffull);
            return cudaSuccess;
        }
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, K, threads, smem);
    if (e != cudaSuccess) return e;
    if (cacheable && per_sm > 0 && per_sm < 256)
        occ[dev].store(key | (uint64_t)per_sm, std::memory_order_relaxed);
    out = (uint64_t)sms * (uint64_t)(per_sm > 0 ? per_sm : 0);
    return cudaSuccess;
}

}  // namespace kvw
