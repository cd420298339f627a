// FP8 E4M3 codec kernels of the MLA graph.
//
// Operations ("mla_graph" module page): convert_bf16_to_fp8_e4m3fn (bf16 ->
// E4M3 codes with a static scale) and the dynamic FP8 scaling used by the
// FP8 branches (here per row: scale = max|x| / 448, codes =
// satfinite_rne(x / scale)).
//
// GB300 design: HBM streaming.  The conversion moves 16 bytes in and 8 bytes
// out per thread and iteration (grid-stride, 4 iterations in flight).  The
// per-row quantiser gives each row to one warp.  Rows of up to 2048 values
// are held in registers (one 16-byte load per lane and 256 columns, all
// issued before any use), so the row is read from HBM once: max |x| as an
// integer maximum of sign-cleared bf16 patterns and one warp redux, the
// scale, then the codes from the registers.  Longer
// rows take a two-pass loop (the second pass re-reads the row from L1/L2).
//
// The per-element division x / scale is the costly part of the quantiser
// (an IEEE divide per value made the first version instruction-bound).  It
// is replaced by one multiply by y = RN(1/scale) and one FMA correction step
// (Markstein's division refinement: P. Markstein, IBM J. Res. Dev. 34(1),
// 1990; also the FMA-based division chapter of Muller et al., Handbook of
// Floating-Point Arithmetic): q0 = RN(x*y), r = x - q0*scale (exact with an
// FMA), q = RN(q0 + r*y), which is the correctly rounded quotient while
// scale, 1/scale and the remainder are normal numbers.  Here x is a bf16
// value and scale = RN(amax / 448) with amax a bf16 magnitude; the path is
// taken for scales in [2^-60, 2^60], where every quotient of magnitude
// >= 2^-14 keeps all three normal, and smaller quotients give an E4M3 zero
// of the right sign whatever their last bits.  Other scales use the IEEE
// divide.  The tests compare every code with a plain division in the CPU
// reference, on rows that hold every bf16 mantissa at every binade that
// matters against every scale mantissa this path can meet.
#include <cstdint>

#include "kvw_device.cuh"

namespace kvw {
namespace {

constexpr uint32_t kThreads = 256;

__global__ void __launch_bounds__(kThreads) convert_kernel(uint2* out, const uint4* in, uint64_t nvec,
                                                           float scale) {
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = ld_stream(in + i + k * stride);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float f[8];
            unpack8(v[k], f);
            store_k8<true>(reinterpret_cast<unsigned char*>(out + i + k * stride), f, scale);
        }
    }
    for (; i < nvec; i += stride) {
        float f[8];
        unpack8(ld_stream(in + i), f);
        store_k8<true>(reinterpret_cast<unsigned char*>(out + i), f, scale);
    }
}

// Scale of a row: max|x| / 448, or 1 for a row of zeros.
__device__ __forceinline__ float row_scale(float amax) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

template <bool REFINED>
__device__ __forceinline__ uint2 quantize8(const uint4& v, float sc, float y) {
    float f[8];
    unpack8(v, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = REFINED ? div_refined(f[e], sc, y) : __fdiv_rn(f[e], sc);
    return pack8_e4m3(f);
}

// One warp per row, VPL 16-byte vectors per lane held in registers
// (cols <= 256 * VPL).
template <int VPL>
__global__ void __launch_bounds__(kThreads) quantize_rows_reg_kernel(
    unsigned char* out, float* scales, const uint16_t* in, uint32_t rows, uint32_t cols,
    int64_t in_stride, int64_t out_stride) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (r >= rows) return;
    const uint4* row = reinterpret_cast<const uint4*>(in + (int64_t)r * in_stride);
    const uint32_t nvec = cols / 8;
    uint4 v[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k)
        v[k] = lane + 32u * k < nvec ? ld_stream(row + lane + 32u * k) : make_uint4(0, 0, 0, 0);
    // max |x| as the largest sign-cleared bf16 pattern (patterns order like
    // magnitudes), a per-halfword unsigned max; a NaN (pattern above
    // infinity) falls back to the float maximum, which ignores it
    uint32_t acc = 0u;
#pragma unroll
    for (int k = 0; k < VPL; ++k)
        acc = __vmaxu2(acc, __vmaxu2(__vmaxu2(v[k].x & 0x7fff7fffu, v[k].y & 0x7fff7fffu),
                                     __vmaxu2(v[k].z & 0x7fff7fffu, v[k].w & 0x7fff7fffu)));
    uint32_t mbits = max(acc & 0xffffu, acc >> 16);
    if (mbits > 0x7f80u) {
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            float f[8];
            unpack8(v[k], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
        }
        mbits = __float_as_uint(amax) >> 16;
    }
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, mbits) << 16);
    const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (lane == 0) scales[r] = sc;
    uint2* orow = reinterpret_cast<uint2*>(out + (int64_t)r * out_stride);
    if (refined_ok(sc)) {
        const float y = __frcp_rn(sc);
#pragma unroll
        for (int k = 0; k < VPL; ++k)
            if (lane + 32u * k < nvec) orow[lane + 32u * k] = quantize8<true>(v[k], sc, y);
    } else {
#pragma unroll
        for (int k = 0; k < VPL; ++k)
            if (lane + 32u * k < nvec) orow[lane + 32u * k] = quantize8<false>(v[k], sc, 0.0f);
    }
}

// Rows longer than 2048 values: max pass, then a second pass over the row.
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(unsigned char* out, float* scales,
                                                                 const uint16_t* in, uint32_t rows,
                                                                 uint32_t cols, int64_t in_stride,
                                                                 int64_t out_stride) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (r >= rows) return;
    const uint4* row = reinterpret_cast<const uint4*>(in + (int64_t)r * in_stride);
    const uint32_t nvec = cols / 8;
    float amax = 0.0f;
    for (uint32_t v = lane; v < nvec; v += 32) {
        float f[8];
        unpack8(ld_table(row + v), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
    }
    const float sc = row_scale(amax);
    if (lane == 0) scales[r] = sc;
    uint2* orow = reinterpret_cast<uint2*>(out + (int64_t)r * out_stride);
    if (refined_ok(sc)) {
        const float y = __frcp_rn(sc);
        for (uint32_t v = lane; v < nvec; v += 32) orow[v] = quantize8<true>(ld_stream(row + v), sc, y);
    } else {
        for (uint32_t v = lane; v < nvec; v += 32)
            orow[v] = quantize8<false>(ld_stream(row + v), sc, 0.0f);
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvw

extern "C" int kvw_convert_bf16_to_fp8_e4m3(void* out, const void* in, uint64_t n, float scale,
                                            cudaStream_t stream) {
    using namespace kvw;
    if (n == 0) return KVW_OK;
    if (!out || !in || n % 8 != 0 || !aligned16(in) ||
        (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
        return KVW_EINVAL;
    if (!(scale > 0.0f && scale < 3.0e38f)) return KVW_EINVAL;
    int sms = 0;
    if (sm_count(sms) != cudaSuccess) return KVW_ECUDA;
    const uint64_t nvec = n / 8;
    uint64_t blocks = (nvec + kThreads - 1) / kThreads;
    const uint64_t cap = (uint64_t)sms * 8;  // 8 resident CTAs per SM, grid-stride beyond
    if (blocks > cap) blocks = cap;
    convert_kernel<<<(uint32_t)blocks, kThreads, 0, stream>>>(static_cast<uint2*>(out),
                                                             static_cast<const uint4*>(in), nvec,
                                                             scale);
    return cudaGetLastError() == cudaSuccess ? KVW_OK : KVW_ECUDA;
}

extern "C" int kvw_quantize_fp8_rows(void* out_codes, float* out_scales, const void* in,
                                     uint32_t rows, uint32_t cols, int64_t in_row_stride,
                                     int64_t out_row_stride, cudaStream_t stream) {
    using namespace kvw;
    if (rows == 0 || cols == 0) return KVW_OK;
    if (!out_codes || !out_scales || !in) return KVW_EINVAL;
    if (cols % 8 != 0 || in_row_stride < (int64_t)cols || in_row_stride % 8 != 0 ||
        out_row_stride < (int64_t)cols || out_row_stride % 8 != 0 || !aligned16(in) ||
        (reinterpret_cast<uintptr_t>(out_codes) & 7u) != 0 ||
        (reinterpret_cast<uintptr_t>(out_scales) & 3u) != 0)
        return KVW_EINVAL;
    const uint32_t rows_per_cta = kThreads / 32;
    const uint32_t grid = (rows + rows_per_cta - 1) / rows_per_cta;
    auto o = static_cast<unsigned char*>(out_codes);
    auto x = static_cast<const uint16_t*>(in);
    const uint32_t vpl = (cols + 255) / 256;  // 16-byte vectors per lane
    if (vpl <= 1)
        quantize_rows_reg_kernel<1><<<grid, kThreads, 0, stream>>>(o, out_scales, x, rows, cols,
                                                                  in_row_stride, out_row_stride);
    else if (vpl <= 2)
        quantize_rows_reg_kernel<2><<<grid, kThreads, 0, stream>>>(o, out_scales, x, rows, cols,
                                                                  in_row_stride, out_row_stride);
    else if (vpl <= 4)
        quantize_rows_reg_kernel<4><<<grid, kThreads, 0, stream>>>(o, out_scales, x, rows, cols,
                                                                  in_row_stride, out_row_stride);
    else if (vpl <= 8)
        quantize_rows_reg_kernel<8><<<grid, kThreads, 0, stream>>>(o, out_scales, x, rows, cols,
                                                                  in_row_stride, out_row_stride);
    else
        quantize_rows_kernel<<<grid, kThreads, 0, stream>>>(o, out_scales, x, rows, cols,
                                                           in_row_stride, out_row_stride);
    return cudaGetLastError() == cudaSuccess ? KVW_OK : KVW_ECUDA;
}
