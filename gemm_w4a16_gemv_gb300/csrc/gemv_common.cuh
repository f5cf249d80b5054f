// Consumer-side building blocks of the M = 1 GEMV kernels (INT4 and FP4):
// activation conversion, code unpacking, the dot-product instructions and the
// multi-row warp reduction.
//
// Arithmetic budget.  A GEMV streaming at HBM speed on 152 SMs must retire
// about 50 weight codes per SM clock.  Measured on sm_103a: the integer dot
// product instructions (dp2a / dp4a) issue at roughly 32 per SM clock, so
// the integer route -- even codes as bytes c, odd codes as bytes 16c (one
// logic op each for four codes), then dp2a against 16-bit activations, four
// dp2a per eight codes -- keeps up with HBM (64 codes per clock), while every
// further dot-product instruction per eight codes costs about an eighth of
// the rate (a second, 8-bit activation part measured 14% slower on the
// 262144 x 3840 GEMV).  The binary16 route (exponent-bias OR, then the mixed
// fma.rn.f32.f16) sustains about 43 codes per clock.
//
// INT4 therefore takes the integer route with one 16-bit integer per
// activation against a power-of-two scale per 128-element group, chosen so
// that a wide range inside a group costs no precision where it matters.  With
// e1 and e3 the exponents of the group's largest and third-largest |x|: if
// e3 >= e1 - 1, e = e1; else e = e3 and the values at or above 2^(e3+1) (the
// largest one or two) are set aside:
//   x = hi * 2^(e-14),  hi = rint(x * 2^(14-e)) in int16     (every other value)
// Values in [2^(e-7), 2^(e+1)) are exact -- so every value at most six binades
// below the third largest's binade -- smaller ones are rounded to a multiple
// of 2^(e-14); the set-aside values ("outliers") enter exactly, as
// binary32 products s * (q - z) * x added per (row, group).  So a group whose
// largest value is 2^14 times the rest keeps the rest at the precision of a
// group without it.  Every product and sum of the integer part is exact in
// 32-bit integers; scale, zero point and activation scale are applied once
// per (row, group) in binary32.
// FP4 codes are not integers (E2M1); they decode exactly to binary16 pairs
// (cvt.rn.f16x2.e2m1x2) and meet binary16 activations, scaled exactly by a
// power of two per 32-element unit, in the mixed-precision FMA.
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

// The eight E2M1 codes of a word -> four f16x2 pairs, h[i] from byte i (low
// half from its low nibble), exact.  One vector move splits the word into
// its bytes, so no shift or mask precedes a conversion.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Largest |x| bit pattern over 32 BF16 values held as 16 words of pairs.
__device__ __forceinline__ uint32_t unit_absmax_bits(const uint32_t (&xb)[16]) {
    uint32_t m2 = 0;  // two packed 16-bit maxima of |x| bit patterns
#pragma unroll
    for (int i = 0; i < 16; ++i) m2 = __vmaxu2(m2, xb[i] & 0x7FFF7FFFu);
    return max(m2 & 0xFFFFu, m2 >> 16);
}

// Exponent e with 2^e <= m < 2^(e+1) for the BF16 magnitude bit pattern m;
// zero gives 14.  Clamped so that 2^(14-e) and 2^(e-14) stay normal binary32
// numbers (subnormal BF16 values read as exponent -127).
__device__ __forceinline__ int exponent_of_absmax(uint32_t m) {
    int e = static_cast<int>(m >> 7) - 127;
    if (m == 0) e = 14;
    e = max(e, -100);
    e = min(e, 113);
    return e;
}

__device__ __forceinline__ int unit_exponent(const uint32_t (&xb)[16]) {
    return exponent_of_absmax(unit_absmax_bits(xb));
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// Load 32 BF16 activations (64 bytes, 16-byte aligned, global memory) as 16
// words of packed pairs: xb[i] = {x[2i], x[2i+1]}.  Cached in L2 only: the
// activation may have been written by the previous kernel of the stream or,
// in a chain of linears, by another CTA of the same launch.
__device__ __forceinline__ void load_x_unit(const uint16_t *x, uint32_t (&xb)[16]) {
    const uint4 *p = reinterpret_cast<const uint4 *>(x);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldcg(p + q);
        xb[4 * q + 0] = v.x;
        xb[4 * q + 1] = v.y;
        xb[4 * q + 2] = v.z;
        xb[4 * q + 3] = v.w;
    }
}

// Round |t| < 2^22 to the nearest integer (ties to even) with one FMA: adding
// 1.5 * 2^23 leaves a binary32 number whose unit in the last place is 1, so
// the sum's low mantissa bits are 2^22 + rint(t).
__device__ __forceinline__ int rint_scaled(float x, float scale) {
    const float r = fmaf(x, scale, 12582912.0f);
    return static_cast<int>(__float_as_uint(r) - 0x4B400000u);
}

__device__ __forceinline__ float bf16_elem(const uint32_t (&xb)[16], int k) {
    return bf16_bits_to_f32((k & 1) ? (xb[k >> 1] >> 16) : (xb[k >> 1] & 0xFFFFu));
}

// d = c + a.lo16 * b.byte0 + a.hi16 * b.byte1   (a: two signed 16-bit values,
// b: unsigned bytes; exact in 32-bit integers)
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// d = c + a.lo16 * b.byte2 + a.hi16 * b.byte3
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t pack_i16x2(int lo, int hi) {
    return (static_cast<uint32_t>(lo) & 0xFFFFu) | (static_cast<uint32_t>(hi) << 16);
}

// The three largest |x| (BF16 magnitude bit patterns) of a set, with the
// position and the signed bits of the first two; ties keep the earlier.
struct Top3 {
    uint32_t a1, a2, a3;  // magnitudes, a1 >= a2 >= a3
    uint32_t p1, p2;      // positions of a1, a2
    uint32_t v1, v2;      // their signed BF16 bits
};

__device__ __forceinline__ void top3_insert(Top3 &t, uint32_t bits, uint32_t pos) {
    const uint32_t m = bits & 0x7FFFu;
    const bool c1 = m > t.a1, c2 = m > t.a2, c3 = m > t.a3;
    t.a3 = c2 ? t.a2 : (c3 ? m : t.a3);
    t.a2 = c1 ? t.a1 : (c2 ? m : t.a2);
    t.p2 = c1 ? t.p1 : (c2 ? pos : t.p2);
    t.v2 = c1 ? t.v1 : (c2 ? bits : t.v2);
    t.a1 = c1 ? m : t.a1;
    t.p1 = c1 ? pos : t.p1;
    t.v1 = c1 ? bits : t.v1;
}

// Top3 of the union of two sets, A listed before B (ties keep A's).
__device__ __forceinline__ Top3 top3_merge(const Top3 &A, const Top3 &B) {
    Top3 t = A;
    top3_insert(t, B.v1, B.p1);
    top3_insert(t, B.v2, B.p2);
    t.a3 = max(t.a3, min(B.a3, t.a2));  // B's third value can only end up third
    return t;
}

// Top3 over the 128 values of a group held by L = 16 / W neighbouring lanes
// (8 W each, positions 8 W (lane mod L) + i); every lane of the L gets the
// same result.  All 32 lanes of the warp call it together.
template <int W>
__device__ __forceinline__ Top3 group_top3(const uint32_t (&xb)[4 * W], int lane) {
    constexpr int L = 16 / W;
    Top3 t = {0u, 0u, 0u, 0u, 0u, 0u, 0u};
    const uint32_t base = 8u * W * static_cast<uint32_t>(lane & (L - 1));
#pragma unroll
    for (int k = 0; k < 8 * W; ++k) top3_insert(t, (k & 1) ? xb[k >> 1] >> 16 : xb[k >> 1] & 0xFFFFu, base + k);
#pragma unroll
    for (int d = 1; d < L; d <<= 1) {
        Top3 o;
        o.a1 = __shfl_xor_sync(0xffffffffu, t.a1, d);
        o.a2 = __shfl_xor_sync(0xffffffffu, t.a2, d);
        o.a3 = __shfl_xor_sync(0xffffffffu, t.a3, d);
        o.p1 = __shfl_xor_sync(0xffffffffu, t.p1, d);
        o.p2 = __shfl_xor_sync(0xffffffffu, t.p2, d);
        o.v1 = __shfl_xor_sync(0xffffffffu, t.v1, d);
        o.v2 = __shfl_xor_sync(0xffffffffu, t.v2, d);
        t = (lane & d) ? top3_merge(o, t) : top3_merge(t, o);  // the lower positions first on both lanes
    }
    return t;
}

// Number of the 2N values (N words of pairs) whose magnitude bit pattern is
// >= thr.
template <int N>
__device__ __forceinline__ int count_at_least(const uint32_t (&xb)[N], uint32_t thr) {
    int c = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) c += ((xb[i] & 0x7FFFu) >= thr) + (((xb[i] >> 16) & 0x7FFFu) >= thr);
    return c;
}

// INT4 activation unit: 32 BF16 values (as 16 words of pairs) and the
// group exponent e -> 16 words of signed 16-bit pairs hi = rint(x *
// 2^(14-e)) in the order the integer dot products meet them: for word m of a
// packed unit (codes 8m..8m+7; its bytes hold codes (8m+2i, 8m+2i+1)), the
// even codes come as bytes (c0, c2, c4, c6) and the odd ones as (16 c1,
// 16 c3, 16 c5, 16 c7), so the pairs are (x0, x2), (x4, x6), (x1, x3),
// (x5, x7).  |hi| <= 32640 for the values below 2^(e+1).  Returns the sum of
// the 32 hi, taken modulo 2^32 (a value at or above 2^(e+1), to be set aside,
// may round to anything: int4_x_drop takes exactly that back out).
__device__ __forceinline__ uint32_t int4_x_unit(const uint32_t (&xb)[16], int e, uint32_t (&xr)[16]) {
    const float inv = pow2f(14 - e);
    uint32_t sum = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        int v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            v[q] = rint_scaled(bf16_elem(xb, 8 * m + q), inv);  // x * inv is exact
            sum += static_cast<uint32_t>(v[q]);
        }
        xr[4 * m + 0] = pack_i16x2(v[0], v[2]);
        xr[4 * m + 1] = pack_i16x2(v[4], v[6]);
        xr[4 * m + 2] = pack_i16x2(v[1], v[3]);
        xr[4 * m + 3] = pack_i16x2(v[5], v[7]);
    }
    return sum;
}

// Take value k (0..31) of a unit converted by int4_x_unit with exponent e
// out again: zero its 16-bit slot and return exactly what int4_x_unit added
// to the sum for it (modulo 2^32).  k = 32: nothing to take out (returns 0).
__device__ __forceinline__ uint32_t int4_x_drop(uint32_t (&xr)[16], const uint32_t (&xb)[16], uint32_t k, int e) {
    const uint32_t m = k >> 3, q = k & 7;  // word m of the unit, value q of the word
    const uint32_t slot = 4 * m + ((q & 1) ? 2 : 0) + ((q >> 2) & 1);  // (x0,x2) (x4,x6) (x1,x3) (x5,x7)
    const bool high = (q >> 1) & 1;                                      // second of its pair
    const uint32_t clear = high ? 0x0000FFFFu : 0xFFFF0000u;
    uint32_t pair = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // static indices and selects: the arrays stay in registers
        const bool at = static_cast<uint32_t>(i) == slot;
        xr[i] &= at ? clear : 0xFFFFFFFFu;
        pair = static_cast<uint32_t>(i) == (k >> 1) ? xb[i] : pair;
    }
    const uint32_t b = (k & 1) ? pair >> 16 : pair & 0xFFFFu;  // its BF16 bits
    return k < 32 ? static_cast<uint32_t>(rint_scaled(bf16_bits_to_f32(b), pow2f(14 - e))) : 0u;
}

// FP4 activation unit: 32 BF16 values -> 16 f16x2 natural pairs (x[2i],
// x[2i+1]) scaled exactly by 2^(14-e) (binary16 holds every BF16 value of the
// unit's top 28 binades exactly); returns pw = 2^(e-14).
__device__ __forceinline__ float fp4_x_unit(const uint32_t (&xb)[16], uint32_t (&xr)[16]) {
    const int e = unit_exponent(xb);
    const float inv = pow2f(14 - e);
#pragma unroll
    for (int q = 0; q < 16; ++q) xr[q] = pack_half2(bf16_elem(xb, 2 * q) * inv, bf16_elem(xb, 2 * q + 1) * inv);
    return pow2f(e - 14);
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
