// Debug dequantisation: packed INT4 / FP4 codes -> binary32 or bfloat16.
// This materialises the weight that the fused kernels keep on chip; it exists
// to pin the unpacking and dequantisation bit-exactly.
#include "common.cuh"
#include "kernels.h"

namespace w4 {
namespace {

// E2M1 code (4 bits) -> value.  The three magnitude bits are placed in the
// two low exponent bits and the top mantissa bit of a binary16 number, the
// sign bit in the binary16 sign: the result is the E2M1 value times 2^-14
// (exponent field 0 gives the subnormal 0 / 0.5 cases).  Multiplying by 2^14
// is exact.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
    const uint16_t h = static_cast<uint16_t>(((c & 7u) << 9) | ((c & 8u) << 12));
    return __half2float(__ushort_as_half(h)) * 16384.0f;
}

// One thread handles 32 consecutive codes (16 packed bytes) of one row.
template <int FMT, int OUT>
__global__ void __launch_bounds__(256)
dequant_kernel(const uint8_t *__restrict__ qw, const uint16_t *__restrict__ s,
               const uint16_t *__restrict__ z, void *__restrict__ out,
               int64_t rows, int64_t K, int group) {
    const int64_t chunks_per_row = K / 32;
    const int64_t total = rows * chunks_per_row;
    const int64_t G = K / group;
    // programmatic dependent launch: the next launch may start; this one's
    // reads and writes follow the previous launch of the stream
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < total;
         c += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = c / chunks_per_row;
        const int64_t k0 = (c % chunks_per_row) * 32;
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(qw + r * (K / 2) + k0 / 2));
        const uint32_t words[4] = {v.x, v.y, v.z, v.w};
        // 32 codes never straddle a group (group is 32 or 128)
        const int64_t gi = r * G + k0 / group;
        const float sf = f16_bits_to_f32(s[gi]);
        // INT4 without zero points is symmetric: the midpoint code 8
        const float zf = (FMT == 0) ? (z ? f16_bits_to_f32(z[gi]) : 8.0f) : 0.0f;
        float w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t code = (words[i / 8] >> (4 * (i % 8))) & 15u;
            if (FMT == 0)
                w[i] = __fmul_rn(__fsub_rn(static_cast<float>(code), zf), sf);
            else
                w[i] = __fmul_rn(e2m1_to_f32(code), sf);
        }
        if (OUT == 0) {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + r * K + k0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                o[i] = make_float4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        } else {
            uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + r * K + k0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t p[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    p[j] = static_cast<uint32_t>(f32_to_bf16_bits(w[8 * i + 2 * j])) |
                           (static_cast<uint32_t>(f32_to_bf16_bits(w[8 * i + 2 * j + 1])) << 16);
                o[i] = make_uint4(p[0], p[1], p[2], p[3]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_dequant(int fmt, const uint8_t *qw, const uint16_t *s,
                           const uint16_t *z, void *out, int out_dtype,
                           int64_t rows, int64_t K, int group, cudaStream_t st,
                           const DeviceInfo &dev) {
    const int64_t total = rows * (K / 32);
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (fmt == 0 && out_dtype == 0) return cudaLaunchKernelEx(&cfg, dequant_kernel<0, 0>, qw, s, z, out, rows, K, group);
    if (fmt == 0) return cudaLaunchKernelEx(&cfg, dequant_kernel<0, 1>, qw, s, z, out, rows, K, group);
    if (out_dtype == 0) return cudaLaunchKernelEx(&cfg, dequant_kernel<1, 0>, qw, s, z, out, rows, K, group);
    return cudaLaunchKernelEx(&cfg, dequant_kernel<1, 1>, qw, s, z, out, rows, K, group);
}

}  // namespace w4
