// FP8 E4M3 codec kernels of the MLA graph.
//
// Operations ("mla_graph" module page): convert_bf16_to_fp8_e4m3fn (bf16 ->
// E4M3 codes with a static scale) and the dynamic FP8 scaling used by the
// FP8 branches (here per row: scale = max|x| / 448, codes =
// satfinite_rne(x / scale)).
//
// GB300 design: HBM streaming.  The conversion moves 16 bytes in and 8 bytes
// out per thread and iteration (grid-stride, 4 iterations in flight).  The
// per-row quantiser gives each row to one warp: a first pass over the row
// finds max|x| (16-byte loads, warp max-reduction), the second pass re-reads
// the row (now in L1/L2) and writes the codes; the scale is stored per row.
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (lane == 0) scales[r] = sc;
    unsigned char* orow = out + (int64_t)r * out_stride;
    for (uint32_t v = lane; v < nvec; v += 32) {
        float f[8];
        unpack8(ld_stream(row + v), f);
        store_k8<true>(orow + 8 * v, f, sc);
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
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVW_ECUDA;
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
    quantize_rows_kernel<<<(rows + rows_per_cta - 1) / rows_per_cta, kThreads, 0, stream>>>(
        static_cast<unsigned char*>(out_codes), out_scales, static_cast<const uint16_t*>(in), rows,
        cols, in_row_stride, out_row_stride);
    return cudaGetLastError() == cudaSuccess ? KVW_OK : KVW_ECUDA;
}
