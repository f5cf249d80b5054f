// Consumer-side building blocks of the M = 1 GEMV kernels (INT4 and FP4):
// activation staging, the mixed-precision multiply-add, code unpacking and
// the multi-row warp reduction.
//
// Arithmetic budget.  On sm_103a the logic / variable-shift / convert pipe
// runs at half the FMA rate, and a GEMV streaming at HBM speed leaves about
// two issue slots per weight element.  The unpack therefore produces two
// codes per logic op as an f16x2 pair, and the multiply-add is the
// mixed-precision fma.rn.f32.f16 (f16 x f16 + f32 -> f32, full rate): every
// product is exact in binary32 and every sum is binary32.
//
// Activations are held as f16 after an exact power-of-two scaling chosen per
// 32-element unit (the largest |x| of the unit lands in [2^14, 2^15)), so the
// BF16 range is never clipped; the scale is undone once per unit.
#pragma once

#include "common.cuh"

namespace w4 {

// d_lo += lo(v) * lo(x); d_hi += hi(v) * hi(x)   (f16 halves, binary32 sums)
__device__ __forceinline__ void mfma_f16x2(uint32_t v, uint32_t x, float &d_lo, float &d_hi) {
    asm("{\n\t.reg .b16 v0, v1, x0, x1;\n\t"
        "mov.b32 {v0, v1}, %2;\n\t"
        "mov.b32 {x0, x1}, %3;\n\t"
        "fma.rn.f32.f16 %0, v0, x0, %0;\n\t"
        "fma.rn.f32.f16 %1, v1, x1, %1;\n\t}"
        : "+f"(d_lo), "+f"(d_hi)
        : "r"(v), "r"(x));
}

// Two E2M1 codes (the low byte of `b`; low nibble = even k) -> their values
// as an f16x2 pair, low half from the low nibble (exact in binary16).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t b) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2)
        : "r"(b));
    return h2;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Exponent e with 2^e <= max|x| < 2^(e+1) over 32 BF16 values (as bits); a
// unit of zeros gives 14.  Clamped so that 2^(14-e) and 2^(e-14) stay normal
// binary32 numbers.
__device__ __forceinline__ int unit_exponent(const uint32_t (&xb)[16]) {
    uint32_t m2 = 0;  // two packed 16-bit maxima of |x| bit patterns
#pragma unroll
    for (int i = 0; i < 16; ++i) m2 = __vmaxu2(m2, xb[i] & 0x7FFF7FFFu);
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    int e = static_cast<int>(m >> 7) - 127;  // BF16 exponent (subnormals read as -127)
    if (m == 0) e = 14;
    e = max(e, -100);
    e = min(e, 113);
    return e;
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// Load 32 BF16 activations (64 bytes, 16-byte aligned) as 16 words of packed
// pairs: xb[i] = {x[2i], x[2i+1]}.
__device__ __forceinline__ void load_x_unit(const uint16_t *x, uint32_t (&xb)[16]) {
    const uint4 *p = reinterpret_cast<const uint4 *>(x);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldg(p + q);
        xb[4 * q + 0] = v.x;
        xb[4 * q + 1] = v.y;
        xb[4 * q + 2] = v.z;
        xb[4 * q + 3] = v.w;
    }
}

__device__ __forceinline__ float bf16_elem(const uint32_t (&xb)[16], int k) {
    return bf16_bits_to_f32((k & 1) ? (xb[k >> 1] >> 16) : (xb[k >> 1] & 0xFFFFu));
}

// Sum of R per-row partials over the 32 lanes of a warp, R in {1, 2, 4}.
// Transposed butterfly: each exchange halves the rows a lane carries, so R
// rows cost R/2 + R/4 + ... + (5 - log2 R) shuffles instead of 5R.  Lanes with
// (lane & (32/R - 1)) == 0 end with the full sum of row reduced_row<R>(lane).
template <int R>
__device__ __forceinline__ float warp_reduce_rows(const float (&p)[R], int lane) {
    if constexpr (R == 1) {
        float v = p[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        return v;
    } else if constexpr (R == 2) {
        const bool up = lane & 16;
        float keep = up ? p[1] : p[0];
        const float send = up ? p[0] : p[1];
        keep += __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
        return keep;
    } else {
        static_assert(R == 4, "rows per thread must be 1, 2 or 4");
        const bool up = lane & 16;
        float k0 = up ? p[2] : p[0], k1 = up ? p[3] : p[1];
        const float s0 = up ? p[0] : p[2], s1 = up ? p[1] : p[3];
        k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
        k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
        const bool up2 = lane & 8;
        float k = up2 ? k1 : k0;
        const float s = up2 ? k0 : k1;
        k += __shfl_xor_sync(0xffffffffu, s, 8);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
        return k;
    }
}

// Row index carried by `lane` after warp_reduce_rows<R>.
template <int R>
__device__ __forceinline__ int reduced_row(int lane) {
    if constexpr (R == 1) return 0;
    else if constexpr (R == 2) return (lane >> 4) & 1;
    else return ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
}

}  // namespace w4
