// Prefill GEMM with INT4 group-128 weights on the tcgen05 tensor cores:
//   Y[m, n] = sum_k X[m, k] * (q[n, k] - z[n, k/128]) * s[n, k/128]
// ("Lab 5: Gemma4 end-to-end inference optimisation": prefill (M > 1) went
// through a Triton dequantiser writing BF16 weights and a cuBLAS GEMM; here the
// weight tile never leaves shared memory, so HBM sees only packed codes).
//
// The dequantisation is split into an exact part that feeds the tensor cores
// and an affine part applied per group to the accumulator:
//   sum_{k in g} X[m,k] (q - z) s = s * A_g[m,n] - s * (128 + z) * S_g[m]
//   A_g[m,n] = sum_{k in g} X[m,k] * (128 + q[n,k])     (BF16 x BF16 MMA)
//   S_g[m]   = sum_{k in g} X[m,k]                       (same MMA: 16 rows of
//                                                         ones below the B tile)
// 128 + q is an integer of at most 8 significant bits, so the B operand is an
// exact BF16 number and X enters as loaded; every product is exact and all
// sums are binary32.
//
// One CTA computes a 128 x 128 output tile over K blocks of 64 (two per group):
//  * CTAs that share an X tile (neighbours along N) form a cluster of C = 4
//    (or 2, 1); all of them need the same 128 x 64 X tile per K block, and
//    128 CTAs reading the same lines make a few L2 slices the bottleneck, so
//    each CTA loads only 128 / C rows and multicasts them to the cluster;
//  * warp 0 (one lane): one bulk copy each of the tile's scale and zero rows;
//    per K block its X rows (TMA, 128-byte swizzle, multicast), and every
//    four K blocks the packed weight bytes of its own tile, 128 bytes of each
//    of the 128 rows per load (TMA, 128-byte swizzle);
//  * warps 8-11: thread n builds row n of the B tile, 64 BF16 values 128 + q
//    from 32 packed bytes with byte permutes, in the same swizzled layout;
//    once per group it also writes the row's (s, -s(128 + z)) into a 4-slot
//    table ring;
//  * warp 1 (one lane): per K block 4 x tcgen05.mma (M=128, N=144, K=16) into
//    the group's TMEM accumulator: columns 0-127 are A_g, column 128 is S_g
//    (a separate N=16 MMA would cost as much as the main one: an instruction
//    takes about as long for N=16 as for N=128);
//    the two accumulator pairs are double-buffered across groups; an X stage
//    is free again only when the MMAs of every CTA of the cluster are done
//    with it, so its commits go to the stage's barrier in all of them;
//  * warps 4-7 and 12-15: per group, read A_g and S_g with tcgen05.ld (warp w
//    serves TMEM lanes 32 (w mod 4) .. +31 and one half of the columns),
//    release the buffers, and accumulate y += s A_g - s (128 + z) S_g in
//    registers; at the end round to BF16 and store Y.
// Every wait is bounded; on timeout the status word is set, each role still
// performs the arrivals the others wait for, and TMEM is always released.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace w4 {
namespace {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int KB_PER_W = 4;           // K blocks per packed-weight load (128 B a row)
constexpr int MAX_XS = 6;             // X ring depth (runtime, from shared memory)
constexpr int WS = 2;                 // packed-weight ring
constexpr int BS = 4;                 // ring of built B tiles
constexpr int TROWS = 16;             // rows of ones appended to each B tile
constexpr int BNX = BN + TROWS;       // MMA N = 144
constexpr int X_BYTES = BM * BK * 2;  // 16 KB BF16 X tile
constexpr int B_BYTES = BNX * BK * 2; // 18 KB BF16 (128 + q) rows, then 16 rows of 1.0
constexpr int W_BYTES = BN * 128;     // 16 KB packed codes, four K blocks
constexpr int TSLOTS = 4;             // group-table ring
constexpr int THREADS = 512;          // 16 warps (2-3 idle)
constexpr int PREP_WARPS = 4;         // warps 8-11
constexpr int EPI_WARPS = 8;          // warps 4-7, 12-15
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_ACC0 = 0, TM_ACC1 = 256;  // 144 columns each; column 128 is S_g
// layout: [B ring][W ring][table][X ring][s tile][z tile][barriers]
constexpr int OFF_B = 0;
constexpr int OFF_W = OFF_B + BS * B_BYTES;
constexpr int OFF_TAB = OFF_W + WS * W_BYTES;
constexpr int OFF_X = ((OFF_TAB + TSLOTS * BN * 8) + 1023) & ~1023;
constexpr int MAX_K = 16384;

struct GemmArgs {
    const uint16_t *s;
    const uint16_t *z;
    uint16_t *Y;
    unsigned int *status;
    int M, N, K, G;
    int sz_bytes;  // bytes of one staged scale (or zero) tile, 16-aligned
    int xs;        // X ring depth
    int csize;     // CTAs per cluster along N (X multicast)
    int off_sz;    // byte offset of the scale tile
};

struct Barriers {
    uint64_t xfull[MAX_XS];   // X tile landed (TMA tx bytes from every cluster CTA)
    uint64_t xempty[MAX_XS];  // MMAs of every cluster CTA done with the stage
    uint64_t wfull[WS];       // packed codes landed (TMA tx bytes)
    uint64_t wempty[WS];      // packed codes read (prep warps)
    uint64_t bready[BS];      // B tile written (prep warps)
    uint64_t bempty[BS];      // MMAs reading the B tile done (commit)
    uint64_t accfull[2];      // group accumulators complete (commit)
    uint64_t accempty[2];     // group accumulators read (epilogue warps)
    uint64_t tfull[TSLOTS];   // group table written (prep warps)
    uint64_t tempty[TSLOTS];  // group table consumed (epilogue warps)
    uint64_t szfull;          // scale/zero tiles landed
    uint64_t done;            // epilogue finished with TMEM
    uint32_t tmem_holder;
};

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// 32x32b.x1: one FP32 column of this warp's 32 TMEM lanes.
__device__ __forceinline__ uint32_t tmem_ld_32x32b_x1(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    return r;
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_int4_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const GemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    // operand tiles need 1024-byte alignment for the 128-byte swizzle
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float2 *table = reinterpret_cast<float2 *>(smem + OFF_TAB);  // [TSLOTS][BN]
    uint16_t *s_tile = reinterpret_cast<uint16_t *>(smem + a.off_sz);
    uint16_t *z_tile = reinterpret_cast<uint16_t *>(smem + a.off_sz + a.sz_bytes);
    Barriers &bar = *reinterpret_cast<Barriers *>(smem + a.off_sz + 2 * a.sz_bytes);
    const int XS = a.xs;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * BM;
    const int nkb = a.K / BK;
    const int ngroups = a.G;
    const int rows_n = min(BN, a.N - n0);  // a multiple of 16

    if (threadIdx.x == 0) {
        for (int i = 0; i < XS; ++i) {
            mbar_init(&bar.xfull[i], 1);
            mbar_init(&bar.xempty[i], a.csize);
        }
        for (int i = 0; i < WS; ++i) {
            mbar_init(&bar.wfull[i], 1);
            mbar_init(&bar.wempty[i], PREP_WARPS);
        }
        for (int i = 0; i < BS; ++i) {
            mbar_init(&bar.bready[i], PREP_WARPS);
            mbar_init(&bar.bempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.accfull[i], 1);
            mbar_init(&bar.accempty[i], EPI_WARPS);
        }
        for (int i = 0; i < TSLOTS; ++i) {
            mbar_init(&bar.tfull[i], PREP_WARPS);
            mbar_init(&bar.tempty[i], EPI_WARPS);
        }
        mbar_init(&bar.szfull, 1);
        mbar_init(&bar.done, EPI_WARPS);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&bar.tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // every CTA's barriers exist before any multicast reaches them
    const uint32_t tmem = bar.tmem_holder;
    const uint32_t crank = cluster_ctarank();
    const uint16_t cmask = static_cast<uint16_t>((1u << a.csize) - 1u);
    const int xrows = BM / a.csize;  // X rows this CTA loads for the cluster

    if (warp == 0) {
        // ------------------------------------------------ packed-weight TMA
        if (lane == 0) {
            tma_prefetch_desc(&tmW);
            const uint64_t pol = policy_evict_first();
            const uint32_t szb = static_cast<uint32_t>(rows_n) * a.G * 2;
            mbar_arrive_expect_tx(&bar.szfull, 2 * szb);
            bulk_g2s(s_tile, a.s + static_cast<size_t>(n0) * a.G, szb, &bar.szfull, pol);
            bulk_g2s(z_tile, a.z + static_cast<size_t>(n0) * a.G, szb, &bar.szfull, pol);
            tma_prefetch_desc(&tmX);
            for (int kb = 0; kb < nkb; ++kb) {
                if (kb % KB_PER_W == 0) {
                    const int wb = kb / KB_PER_W, ws = wb % WS;
                    if (wb >= WS && !mbar_wait(&bar.wempty[ws], ((wb / WS) - 1) & 1, a.status)) break;
                    mbar_arrive_expect_tx(&bar.wfull[ws], W_BYTES);
                    tma_load_2d(smem + OFF_W + ws * W_BYTES, &tmW, wb * 128, n0, &bar.wfull[ws]);
                }
                const int st = kb % XS;
                if (kb >= XS && !mbar_wait(&bar.xempty[st], ((kb / XS) - 1) & 1, a.status)) break;
                mbar_arrive_expect_tx(&bar.xfull[st], X_BYTES);  // the whole tile, from all slices
                unsigned char *dst = smem + OFF_X + st * X_BYTES + static_cast<int>(crank) * xrows * 128;
                if (a.csize > 1)
                    tma_load_2d_multicast(dst, &tmX, kb * BK, m0 + static_cast<int>(crank) * xrows, &bar.xfull[st], cmask);
                else
                    tma_load_2d(dst, &tmX, kb * BK, m0, &bar.xfull[st]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_main = idesc_kind_f16(BM, BNX, 1u);  // BF16, N = 144
            bool ok = true;
            for (int g = 0; ok && g < ngroups; ++g) {
                const int ab = g & 1;
                if (g >= 2 && !mbar_wait(&bar.accempty[ab], ((g >> 1) - 1) & 1, a.status)) break;
                tc_fence_after();
                const uint32_t t_acc = tmem + (ab ? TM_ACC1 : TM_ACC0);
                for (int kk = 0; kk < 2; ++kk) {
                    const int kb = 2 * g + kk;
                    const int st = kb % XS, bs = kb % BS;
                    if (!mbar_wait(&bar.xfull[st], (kb / XS) & 1, a.status) ||
                        !mbar_wait(&bar.bready[bs], (kb / BS) & 1, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + OFF_X + st * X_BYTES);
                    const uint32_t b_addr = smem_u32(smem + OFF_B + bs * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        umma_f16(t_acc, smem_desc_sw128_kmajor(a_addr + 32 * k), smem_desc_sw128_kmajor(b_addr + 32 * k),
                                 idesc_main, (kk | k) != 0);
                    }
                    if (a.csize > 1)
                        umma_commit_multicast(&bar.xempty[st], cmask);
                    else
                        umma_commit(&bar.xempty[st]);
                    umma_commit(&bar.bempty[bs]);
                }
                if (!ok) break;
                umma_commit(&bar.accfull[ab]);
            }
            // Only after a timeout: one more commit so that the epilogue's wait
            // also ends once the MMAs already issued have completed.
            if (!ok) umma_commit(&bar.accfull[0]);
        }
        __syncwarp();
        mbar_wait(&bar.done, 0, a.status);
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    } else if (warp >= 8 && warp < 12) {
        // -------------------------------------------------- B-tile builders
        const int n = threadIdx.x - 256;  // W row of this thread
        const bool row_ok = n < rows_n;
        // rows 128-143 of every B stage: BF16 1.0 (every chunk alike, swizzle moot)
        for (int b = 0; b < BS; ++b)
            reinterpret_cast<uint4 *>(smem + OFF_B + b * B_BYTES + BN * 128)[n] =
                make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        fence_proxy_async_smem();
        bool ok = mbar_wait(&bar.szfull, 0, a.status);
        unsigned char *b_row_base = smem + OFF_B + (n >> 3) * 1024 + (n & 7) * 128;
        for (int kb = 0; ok && kb < nkb; ++kb) {
            const int bs = kb % BS;
            if ((kb & 1) == 0) {
                // this group's (s, -s (128 + z)) for row n into the table ring
                const int g = kb >> 1, slot = g % TSLOTS;
                if (g >= TSLOTS && !mbar_wait(&bar.tempty[slot], ((g / TSLOTS) - 1) & 1, a.status)) break;
                const float sf = row_ok ? f16_bits_to_f32(s_tile[n * a.G + g]) : 0.0f;
                const float zf = row_ok ? f16_bits_to_f32(z_tile[n * a.G + g]) : 0.0f;
                table[slot * BN + n] = make_float2(sf, -sf * (128.0f + zf));
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.tfull[slot]);
            }
            const int wb = kb / KB_PER_W, kk = kb % KB_PER_W, ws = wb % WS;
            if (kk == 0 && !mbar_wait(&bar.wfull[ws], (wb / WS) & 1, a.status)) break;
            if (kb >= BS && !mbar_wait(&bar.bempty[bs], ((kb / BS) - 1) & 1, a.status)) break;
            // row n of the packed stage: 16-byte chunk c sits at c ^ (n mod 8)
            const unsigned char *wrow = smem + OFF_W + ws * W_BYTES + n * 128;
            const uint4 p0 = *reinterpret_cast<const uint4 *>(wrow + (((2 * kk) ^ (n & 7)) << 4));
            const uint4 p1 = *reinterpret_cast<const uint4 *>(wrow + (((2 * kk + 1) ^ (n & 7)) << 4));
            const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            unsigned char *b_row = b_row_base + bs * B_BYTES;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // codes 8j..8j+7 (code i at bits 4i..4i+3) -> BF16 128 + q,
                // which is the byte q under the byte 0x43
                const uint32_t w = words[j];
                const uint32_t lo = w & 0x0F0F0F0Fu;         // q0 q2 q4 q6
                const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // q1 q3 q5 q7
                const uint32_t q0123 = __byte_perm(lo, hi, 0x5140);
                const uint32_t q4567 = __byte_perm(lo, hi, 0x7362);
                const uint4 out = make_uint4(__byte_perm(q0123, 0x43434343u, 0x4140), __byte_perm(q0123, 0x43434343u, 0x4342),
                                             __byte_perm(q4567, 0x43434343u, 0x4140), __byte_perm(q4567, 0x43434343u, 0x4342));
                // 16-byte chunk j of row n goes to chunk j ^ (n mod 8)
                *reinterpret_cast<uint4 *>(b_row + ((j ^ (n & 7)) << 4)) = out;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar.bready[bs]);
                if (kk == KB_PER_W - 1 || kb == nkb - 1) mbar_arrive(&bar.wempty[ws]);
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ group epilogue
        const int qd = warp & 3;                 // TMEM lane quarter
        const int hc = warp >= 12 ? 1 : 0;       // column half
        const int row = qd * 32 + lane;          // output row in the tile
        const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
        float y[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) y[j] = 0.0f;
        bool ok = true;
        for (int g = 0; ok && g < ngroups; ++g) {
            const int ab = g & 1, slot = g % TSLOTS;
            if (!mbar_wait(&bar.accfull[ab], (g >> 1) & 1, a.status) ||
                !mbar_wait(&bar.tfull[slot], (g / TSLOTS) & 1, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t t_acc = tmem + lane_off + (ab ? TM_ACC1 : TM_ACC0) + hc * 64;
            const float ssum = __uint_as_float(tmem_ld_32x32b_x1(tmem + lane_off + (ab ? TM_ACC1 : TM_ACC0) + BN));
            const float2 *tab = table + slot * BN + hc * 64;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_acc + c * 32, r);
                tmem_ld_wait();
                if (c == 1) {
                    // both halves are in registers: hand the buffers back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar.accempty[ab]);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float2 sc = tab[c * 32 + j];
                    y[c * 32 + j] = fmaf(sc.x, __uint_as_float(r[j]), fmaf(sc.y, ssum, y[c * 32 + j]));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.tempty[slot]);
        }
        const int m = m0 + row;
        if (ok && m < a.M) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.Y + static_cast<size_t>(m) * a.N + n0 + hc * 64);
            const int valid_cols = rows_n - hc * 64;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q * 8 < valid_cols) {
                    uint4 o;
                    o.x = bf16x2_rn(y[8 * q + 0], y[8 * q + 1]);
                    o.y = bf16x2_rn(y[8 * q + 2], y[8 * q + 3]);
                    o.z = bf16x2_rn(y[8 * q + 4], y[8 * q + 5]);
                    o.w = bf16x2_rn(y[8 * q + 6], y[8 * q + 7]);
                    dst[q] = o;
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.done);
    }
    // no CTA leaves while cluster peers may still signal or fill its memory
    cluster_sync();
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
    const unsigned gx = static_cast<unsigned>((N + BN - 1) / BN), gy = static_cast<unsigned>((M + BM - 1) / BM);
    const int csize = (gx % 4 == 0) ? 4 : (gx % 2 == 0) ? 2 : 1;
    CUtensorMap tmX, tmW;
    {
        // X as BF16 [M, K]; box of 64 (one K block) x 128/csize rows, 128-byte swizzle
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {BK, static_cast<cuuint32_t>(BM / csize)};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(X), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // packed codes as bytes [N, K/2]; box of 128 bytes (four K blocks) x 128 rows
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
        const cuuint32_t box[2] = {128, BN};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(qw), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    GemmArgs a;
    a.csize = csize;
    a.s = s;
    a.z = z;
    a.Y = Y;
    a.status = status;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.G = static_cast<int>(K / 128);
    a.sz_bytes = (BN * a.G * 2 + 15) & ~15;
    // as many X stages as shared memory allows (3 .. MAX_XS)
    const int fixed = 1024 + OFF_X + 2 * a.sz_bytes + static_cast<int>(sizeof(Barriers)) + 16;
    int xs = (dev.max_smem_optin - fixed) / X_BYTES;
    if (xs > MAX_XS) xs = MAX_XS;
    if (xs < 2) return cudaErrorNotSupported;
    a.xs = xs;
    a.off_sz = OFF_X + xs * X_BYTES;
    const int smem = 1024 + a.off_sz + 2 * a.sz_bytes + static_cast<int>(sizeof(Barriers));
    static int configured[64] = {0};
    const int d = dev.device & 63;
    if (configured[d] < smem) {
        cudaError_t e = cudaFuncSetAttribute(gemm_int4_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[d] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, gy, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_int4_tc_kernel, tmX, tmW, a);
}

}  // namespace w4
