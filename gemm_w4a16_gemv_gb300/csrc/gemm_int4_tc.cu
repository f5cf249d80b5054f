// Prefill GEMM with INT4 group-128 weights on the tcgen05 tensor cores:
//   Y[m, n] = sum_k X[m, k] * (q[n, k] - z[n, k/128]) * s[n, k/128]
// ("Lab 5: Gemma4 end-to-end inference optimisation": prefill (M > 1) went
// through a Triton dequantiser writing BF16 weights and a cuBLAS GEMM; here the
// dequantised tile never leaves shared memory, so HBM sees only packed codes).
//
// One CTA computes a 128 x 128 output tile, looping over K in blocks of 64:
//  * warp 0 (one lane) loads the X tile (TMA, 128-byte swizzle) and the packed
//    weight bytes of the tile (TMA, 32 B x 128 rows) into a 4-stage ring, and
//    once per CTA the tile's scale and zero rows (one bulk copy each);
//  * warps 4-11 prepare both operands of each block in shared memory: thread
//    (n, h) takes half h of row n -- it converts half of the 16-byte chunks of
//    X row n in place from BF16 to F16, and turns 32 codes of W row n into
//    binary32 W = (q - z) * s with one FMA per code (exact for integer zero
//    points), rounded once to F16 and stored in the K-major 128-byte-swizzled
//    layout the MMA reads; then it fences the async proxy and arrives;
//  * warp 1 (one lane) issues 4 x tcgen05.mma kind::f16 (F16 x F16 -> F32,
//    M=128, N=128, K=16) per block into a TMEM accumulator and commits the
//    stage back to the producer;
//  * warps 4-7 finally read the accumulator with tcgen05.ld (each warp its
//    32-lane quarter), round to BF16 and store Y.
// F16 rather than BF16 operands: a BF16 weight keeps 8 significant bits, and
// at K = 3840 its rounding alone moves outputs near zero by more than the
// accepted 2e-2 absolute; F16 keeps 11 bits.  An activation outside the F16
// range (|x| >= 65520) cannot be represented: it sets kDevRange.
// Every wait is bounded; on timeout the status word is set and each role still
// performs the arrivals the others wait for, and TMEM is always released.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace w4 {
namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB X tile (BF16 as loaded, F16 after conversion)
constexpr int B_BYTES = BN * BK * 2;  // 16 KB F16 W tile
constexpr int P_BYTES = BN * BK / 2;  // 4 KB packed codes
constexpr int THREADS = 384;   // 12 warps: producer, MMA, 2 idle, 8 operand warps
constexpr int PREP_WARPS = 8;
constexpr uint32_t TMEM_COLS = BN;    // 128 FP32 columns
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_P = OFF_B + STAGES * B_BYTES;
constexpr int OFF_SZ = OFF_P + STAGES * P_BYTES;
constexpr int MAX_K = 16384;

struct GemmArgs {
    const uint16_t *s;
    const uint16_t *z;
    uint16_t *Y;
    unsigned int *status;
    int M, N, K, G;
    int sz_bytes;  // bytes of one staged scale (or zero) tile, 16-aligned
};

struct Barriers {
    uint64_t full[STAGES];    // X + packed tile landed (TMA tx bytes)
    uint64_t bready[STAGES];  // F16 X and W tiles written (8 warps)
    uint64_t empty[STAGES];   // MMAs of the stage done (commit)
    uint64_t szfull;          // scale/zero tiles landed
    uint64_t accfull;         // accumulator complete (commit)
    uint64_t done;            // epilogue finished reading TMEM (4 warps)
    uint32_t tmem_holder;
};

__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_int4_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const GemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    // operand tiles need 1024-byte alignment for the 128-byte swizzle
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint16_t *s_tile = reinterpret_cast<uint16_t *>(smem + OFF_SZ);
    uint16_t *z_tile = reinterpret_cast<uint16_t *>(smem + OFF_SZ + a.sz_bytes);
    Barriers &bar = *reinterpret_cast<Barriers *>(smem + OFF_SZ + 2 * a.sz_bytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * BM;
    const int nkb = a.K / BK;
    const int rows_n = min(BN, a.N - n0);  // a multiple of 16

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bar.full[s], 1);
            mbar_init(&bar.bready[s], PREP_WARPS);
            mbar_init(&bar.empty[s], 1);
        }
        mbar_init(&bar.szfull, 1);
        mbar_init(&bar.accfull, 1);
        mbar_init(&bar.done, 4);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&bar.tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmW);
            const uint64_t pol = policy_evict_first();
            const uint32_t szb = static_cast<uint32_t>(rows_n) * a.G * 2;
            mbar_arrive_expect_tx(&bar.szfull, 2 * szb);
            bulk_g2s(s_tile, a.s + static_cast<size_t>(n0) * a.G, szb, &bar.szfull, pol);
            bulk_g2s(z_tile, a.z + static_cast<size_t>(n0) * a.G, szb, &bar.szfull, pol);
            for (int kb = 0; kb < nkb; ++kb) {
                const int st = kb % STAGES;
                if (kb >= STAGES && !mbar_wait(&bar.empty[st], ((kb / STAGES) - 1) & 1, a.status)) break;
                mbar_arrive_expect_tx(&bar.full[st], A_BYTES + P_BYTES);
                tma_load_2d(smem + OFF_A + st * A_BYTES, &tmX, kb * BK, m0, &bar.full[st]);
                tma_load_2d(smem + OFF_P + st * P_BYTES, &tmW, kb * BK / 2, n0, &bar.full[st]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_kind_f16(BM, BN, 0u);  // F16 operands
            for (int kb = 0; kb < nkb; ++kb) {
                const int st = kb % STAGES;
                const uint32_t par = (kb / STAGES) & 1;
                if (!mbar_wait(&bar.full[st], par, a.status)) break;
                if (!mbar_wait(&bar.bready[st], par, a.status)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + OFF_A + st * A_BYTES);
                const uint32_t b_addr = smem_u32(smem + OFF_B + st * B_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_f16(tmem, smem_desc_sw128_kmajor(a_addr + 32 * k), smem_desc_sw128_kmajor(b_addr + 32 * k),
                              idesc, (kb | k) != 0);
                umma_commit(&bar.empty[st]);
            }
            umma_commit(&bar.accfull);  // after everything issued, on every path
        }
        __syncwarp();
        mbar_wait(&bar.done, 0, a.status);
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    } else if (warp >= 4) {
        // ------------------------------------------- operands, then epilogue
        const int t = threadIdx.x - 128;
        const int n = t & (BN - 1);  // W row of this thread (and TMEM lane in warps 4-7)
        const int h = t >> 7;        // which half of the row's codes / chunks
        const bool row_ok = n < rows_n;
        bool ok = mbar_wait(&bar.szfull, 0, a.status);
        float2 c_ev = make_float2(0.f, 0.f), c_12 = c_ev, c_16 = c_ev;
        float2 s2 = c_ev;
        uint32_t xmax = 0;  // two packed maxima of |x| bit patterns (BF16)
        unsigned char *b_row_base = smem + OFF_B + (n >> 3) * 1024 + (n & 7) * 128;
        for (int kb = 0; ok && kb < nkb; ++kb) {
            const int st = kb % STAGES;
            if (!mbar_wait(&bar.full[st], (kb / STAGES) & 1, a.status)) {
                ok = false;
                break;
            }
            if ((kb & 1) == 0) {
                // new group: W = (128+q)*s - (128+z)*s or (2048+q)*s - (2048+z)*s
                const int g = kb >> 1;
                const float sf = row_ok ? f16_bits_to_f32(s_tile[n * a.G + g]) : 0.0f;
                const float zf = row_ok ? f16_bits_to_f32(z_tile[n * a.G + g]) : 0.0f;
                const float c128 = -(128.0f + zf) * sf, c2048 = -(2048.0f + zf) * sf;
                s2 = make_float2(sf, sf);
                c_ev = make_float2(c2048, c128);  // (12-bit slot, 16-bit slot)
                c_12 = make_float2(c2048, c2048);
                c_16 = make_float2(c128, c128);
            }
            {
                // X row n of this block: BF16 -> F16 in place.  Conversion is
                // elementwise, so each 16-byte chunk is converted where it lies;
                // the chunk visited is rotated by the row so that the 8 lanes of
                // a shared-memory phase touch 8 different bank groups.
                uint4 *xr = reinterpret_cast<uint4 *>(smem + OFF_A + st * A_BYTES + (n >> 3) * 1024 + (n & 7) * 128);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = (q + 4 * h + n) & 7;
                    uint4 v = xr[c];
                    xmax = __vmaxu2(xmax, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                                   __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
                    v.x = f16x2_rn(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u));
                    v.y = f16x2_rn(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
                    v.z = f16x2_rn(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u));
                    v.w = f16x2_rn(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
                    xr[c] = v;
                }
            }
            const uint4 p0 = *reinterpret_cast<const uint4 *>(smem + OFF_P + st * P_BYTES + n * 32 + h * 16);
            const uint32_t words[4] = {p0.x, p0.y, p0.z, p0.w};
            unsigned char *b_row = b_row_base + st * B_BYTES;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * h + jj;  // 16-byte chunk (8 codes) of the row
                // codes k = 8j .. 8j+7 of this block; code i sits at bits 4i..4i+3.
                // Binary32 with the code at mantissa bits 12-15 (exponent of
                // 2048) is 2048 + q; at bits 16-19 (exponent of 128) 128 + q.
                const uint32_t w = words[jj];
                const uint32_t l12 = w << 12, l4 = w << 4, r4 = w >> 4, r12 = w >> 12;
                const float2 v01 = make_float2(__uint_as_float((l12 & 0x0000F000u) | 0x45000000u),
                                               __uint_as_float((l12 & 0x000F0000u) | 0x43000000u));
                const float2 v23 = make_float2(__uint_as_float((l4 & 0x0000F000u) | 0x45000000u),
                                               __uint_as_float((w & 0x0000F000u) | 0x45000000u));
                const float2 v45 = make_float2(__uint_as_float((w & 0x000F0000u) | 0x43000000u),
                                               __uint_as_float((r4 & 0x000F0000u) | 0x43000000u));
                const float2 v67 = make_float2(__uint_as_float((r12 & 0x0000F000u) | 0x45000000u),
                                               __uint_as_float((r12 & 0x000F0000u) | 0x43000000u));
                const float2 w01 = __ffma2_rn(v01, s2, c_ev);
                const float2 w23 = __ffma2_rn(v23, s2, c_12);
                const float2 w45 = __ffma2_rn(v45, s2, c_16);
                const float2 w67 = __ffma2_rn(v67, s2, c_ev);
                const uint4 out = make_uint4(f16x2_rn(w01.x, w01.y), f16x2_rn(w23.x, w23.y),
                                             f16x2_rn(w45.x, w45.y), f16x2_rn(w67.x, w67.y));
                // 16-byte chunk j of row n goes to chunk j ^ (n mod 8)
                *reinterpret_cast<uint4 *>(b_row + ((j ^ (n & 7)) << 4)) = out;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.bready[st]);
        }
        // BF16 0x4780 = 65536: from there on F16 rounds to infinity
        if (max(xmax & 0xFFFFu, xmax >> 16) > 0x477Fu) atomicOr(a.status, kDevRange);
        if (warp >= 8) return;  // warps 8-11: operands only
        // epilogue (warps 4-7): accumulator lane n = output row m0 + n
        if (mbar_wait(&bar.accfull, 0, a.status)) {
            tc_fence_after();
            const int m = m0 + n;
            const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_lane + c * 32, r);
                tmem_ld_wait();
                if (m < a.M) {
                    uint4 *dst = reinterpret_cast<uint4 *>(a.Y + static_cast<size_t>(m) * a.N + n0 + c * 32);
                    const int valid_cols = rows_n - c * 32;  // columns of the tile inside N
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (q * 8 < valid_cols) {
                            uint4 o;
                            o.x = bf16x2_rn(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]));
                            o.y = bf16x2_rn(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
                            o.z = bf16x2_rn(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
                            o.w = bf16x2_rn(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
                            dst[q] = o;
                        }
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.done);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

cudaError_t launch_gemm_int4(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const uint16_t *z,
                             uint16_t *Y, int64_t M, int64_t N, int64_t K, cudaStream_t st, unsigned int *status,
                             const DeviceInfo &dev) {
    if (K > MAX_K) return cudaErrorNotSupported;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap tmX, tmW;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {BK, BM};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(X), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
        const cuuint32_t box[2] = {BK / 2, BN};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(qw), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    GemmArgs a;
    a.s = s;
    a.z = z;
    a.Y = Y;
    a.status = status;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.G = static_cast<int>(K / 128);
    a.sz_bytes = (BN * a.G * 2 + 15) & ~15;
    const int smem = 1024 + OFF_SZ + 2 * a.sz_bytes + static_cast<int>(sizeof(Barriers));
    static int configured[64] = {0};
    const int d = dev.device & 63;
    if (configured[d] < smem) {
        cudaError_t e = cudaFuncSetAttribute(gemm_int4_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[d] = smem;
    }
    const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>((M + BM - 1) / BM));
    gemm_int4_tc_kernel<<<grid, THREADS, smem, st>>>(tmX, tmW, a);
    return cudaGetLastError();
}

}  // namespace w4
