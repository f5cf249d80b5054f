// Prefill GEMM with INT4 group-128 weights on the tcgen05 tensor cores:
//   Y[m, n] = sum_k X[m, k] * (q[n, k] - z[n, k/128]) * s[n, k/128]
// ("Lab 5: Gemma4 end-to-end inference optimisation": prefill (M > 1) went
// through a Triton dequantiser writing BF16 weights and a cuBLAS GEMM; here the
// dequantised weight tile never leaves the SM, so HBM sees only packed codes).
//
// Operands are binary16, so that one FP32 accumulator runs over all of K:
//  * each weight is formed once as fl16(fl16(q - z) * s): q - z is exact for
//    an integer zero point (GPTQ-style codes), so the weight carries one
//    rounding, a relative error of at most 2^-11 (the BF16 weights of the
//    two-pass path carry 2^-9);
//  * each row of X is scaled by a power of two into binary16 by a pre-pass
//    (largest |x| of the row in [2^14, 2^15): every BF16 value within 2^28
//    of that maximum is exact), the epilogue undoes the scale per row.
// The pre-pass also permutes K within each block of 8 to 0,4,1,5,2,6,3,7:
// a 32-bit word of packed codes then yields its four binary16 pairs
// (codes i and i + 4) with one shift, one mask and two pair instructions
// each, and the MMA pairs them with the same permuted X columns.
//
// One CTA computes 128 weight rows n x NT token rows m (NT = 256, or M
// rounded up to 16 when smaller), K in chunks of 64 (four MMAs of K = 16):
//  * warp 0 (one lane): the packed codes, 128 rows x 128 bytes (256 K) per
//    TMA load (128-byte swizzle), on a ring of WS stages;
//  * warp 1 (one lane): per chunk the X tile, NT rows x 64 binary16 (one
//    TMA box, 128-byte swizzle), on a ring of XS stages;
//  * warp 0 also copies the tile's scale and zero rows into shared memory
//    (one bulk copy each);
//  * warps 8-23: per chunk (group of four warps c mod 4, TMEM lane
//    quarter warp mod 4) thread r turns the 64 codes of weight row r into
//    32 binary16 pairs in the chunk's TMEM operand stage (one of 8);
//  * warps 2-5: MMA issuers.  MMAs issued by one thread run one after
//    another at roughly 100-150 SM cycles each even at N = 16, while MMAs
//    issued by different warps into different accumulators overlap, so
//    tiles of NT <= 64 (<= 128) token rows use 4 (2) issuers, issuer j
//    taking the chunks c = j mod n_iss into accumulator j; NT = 256 uses
//    one (a K = 16 MMA of N = 256 keeps the tensor pipe busy by itself);
//  * at the end warps 8-23 sum the issuers' accumulators, undo the row
//    scale of X, round to BF16 and store Y (for N % 8 == 0 through a
//    shared-memory tile in the idle X ring and one TMA store).
// Every wait is bounded; on a timeout the status word is set, each role
// still performs the arrivals the others wait for, and tensor memory is
// released only after every MMA issued has completed.
#include "common.cuh"
#include "gemv_common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

#include <cstring>
#include <mutex>

namespace w4 {
namespace {

constexpr int BR = 128;               // weight rows per CTA (TMEM lanes, the MMA's M)
constexpr int NT_MAX = 256;           // token rows per CTA at most (the MMA's N)
constexpr int CK = 64;                // K per chunk
constexpr int GK = 128;               // K per quantisation group
constexpr int WS = 3;                 // packed-code stages, 256 K each
constexpr int W_STAGE = BR * 128;     // 16 KB
constexpr int XS_MAX = 8;             // X stages: as many as fit (a multiple of the issuer count)
constexpr int SMEM_BUDGET = 226 * 1024;
constexpr int AP = 8;                 // TMEM operand stages, 32 columns (64 K) each
constexpr int MAX_ISS = 4;
constexpr int THREADS = 768;          // 24 warps
constexpr int ISS0 = 2;               // first issuer warp
constexpr int BW0 = 8;                // first builder warp
constexpr int NBW = 16;               // builder warps: groups of 4 (one per TMEM lane quarter)
constexpr int BG = NBW / 4;           // builder groups: chunk c is built by group c mod BG
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_ACC = 0;        // accumulators: n_iss x NT <= 256 columns
constexpr uint32_t TM_A = 256;        // operand stages after them
constexpr int PRE_THREADS = 256;
constexpr int PRE_BLOCKS = 8;  // at most 8 blocks of 8 values of X per pre-pass thread: K <= 16384

struct GemmF16Args {
    const uint16_t *s;
    const uint16_t *z;       // null: symmetric (z = 8)
    const float *rowscale;   // [M] 2^(e - 14) of each X row
    uint16_t *Y;
    unsigned int *status;
    int M, N, K, G, nt, ntn;  // ntn: tiles along N
    int xs_n;                 // X ring depth
    int off_w, off_sz, off_bar;  // shared-memory offsets (X ring at 0)
    int y_tma;                // Y written by one TMA store per tile (N % 8 == 0)
    unsigned int inject;
    int tiles_full;           // CTAs 0 .. tiles_full - 1: whole tiles (numbered N fastest)
    int nsplit, cps;          // CTA tiles_full + nsplit x + y: chunks [y cps, y cps + cps) of K of
                              // tile tiles_full + x (cps a multiple of 4)
    float *part;              // their binary32 partial sums [x][y][m][r]
};

struct Barriers {
    uint64_t xfull[XS_MAX], xempty[XS_MAX];
    uint64_t wfull[WS], wempty[WS];
    uint64_t aready[AP], aempty[AP];
    uint64_t szfull;    // the scale (and zero) tile landed
    uint64_t accfull;   // every issuer's MMAs completed (n_iss arrivals)
    uint64_t done;      // builders finished reading tensor memory
    uint32_t tmem_holder;
};

// ---------------------------------------------------------------- pre-pass
// One CTA per row of X: the row's largest |x| (BF16 magnitude bits order as
// the values), then binary16 x * 2^(14 - e) in the permuted K order.  The
// row is read once: each thread keeps its NB blocks of 8 values in registers
// (K / 8 <= NB x PRE_THREADS), all loads in flight together; NB follows K so
// that short rows keep few registers (and many CTAs per SM).
template <int NB>
__global__ void __launch_bounds__(PRE_THREADS) x16_prepass_kernel(const uint16_t *__restrict__ X, int K,
                                                                  uint16_t *__restrict__ Xh, float *rowscale) {
    const int m = blockIdx.x;
    pdl_launch_dependents();  // the GEMM's CTAs may start; they wait for this grid before reading
    pdl_wait();               // X (and the scratch's previous user) follow the stream order
    const uint4 *x = reinterpret_cast<const uint4 *>(X + static_cast<int64_t>(m) * K);
    uint4 *xh = reinterpret_cast<uint4 *>(Xh + static_cast<int64_t>(m) * K);
    const int nb = K / 8;
    __shared__ uint32_t red[PRE_THREADS / 32];
    uint4 xv[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        const int b = threadIdx.x + j * PRE_THREADS;
        xv[j] = b < nb ? x[b] : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t mx = 0;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0;
#pragma unroll
    for (int w = 0; w < PRE_THREADS / 32; ++w) mx = max(mx, red[w]);
    const int e = exponent_of_absmax(mx);  // 2^e <= max|x| < 2^(e+1)
    const float inv = pow2f(14 - e);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        const int b = threadIdx.x + j * PRE_THREADS;
        if (b >= nb) break;
        const uint4 v = xv[j];
        // values 0..7 of the block: v.x = {0, 1}, v.y = {2, 3}, v.z = {4, 5}, v.w = {6, 7}
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu) * inv;
            f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16) * inv;
        }
        // positions 0..7 hold values 0, 4, 1, 5, 2, 6, 3, 7
        uint4 o;
        o.x = pack_half2(f[0], f[4]);
        o.y = pack_half2(f[1], f[5]);
        o.z = pack_half2(f[2], f[6]);
        o.w = pack_half2(f[3], f[7]);
        xh[b] = o;
    }
    if (threadIdx.x == 0) rowscale[m] = pow2f(e - 14);
}

// ------------------------------------------------------------------- GEMM
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

template <bool SYM>
__global__ void __launch_bounds__(THREADS, 1)
gemm_int4_f16_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmY, const GemmF16Args a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint16_t *s_t = reinterpret_cast<uint16_t *>(smem + a.off_sz);  // [BR][G] binary16 scales of the tile's rows
    uint16_t *z_t = s_t + BR * a.G;                                 // [BR][G] zero points
    float *rs_t = reinterpret_cast<float *>(smem + a.off_bar - NT_MAX * 4);  // row scales of the tile's X rows
    Barriers &bar = *reinterpret_cast<Barriers *>(smem + a.off_bar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's tile and chunks of K, [c0, c0 + nch) with c0 a multiple of 4
    // (whole packed-code stages); ring slots and phases count from c0
    const int b = static_cast<int>(blockIdx.x);
    const bool partial = b >= a.tiles_full;  // uniform over the CTA
    const int part_id = b - a.tiles_full;    // index of the partial sums (partial CTAs)
    const int tile = partial ? a.tiles_full + part_id / a.nsplit : b;
    const int c0 = partial ? (part_id % a.nsplit) * a.cps : 0;
    const int nch = partial ? min(a.cps, a.K / CK - c0) : a.K / CK;
    const int tn = tile % a.ntn, tm = tile / a.ntn;  // N fastest: neighbours share X
    const int n0 = tn * BR, m0 = tm * a.nt;
    const int nt = a.nt;
    const bool y_tma = a.y_tma && !partial;
    int n_iss = nt <= 64 ? MAX_ISS : (nt <= 128 ? 2 : 1);
    n_iss = n_iss < nch ? n_iss : nch;
    const int xs_n = a.xs_n;  // a multiple of 4 or of n_iss: each issuer waits on its own stages only
    const int x_stage = nt * 128;

    if (threadIdx.x == 0) {
        for (int i = 0; i < xs_n; ++i) {
            mbar_init(&bar.xfull[i], 1);
            mbar_init(&bar.xempty[i], 1);
        }
        for (int i = 0; i < WS; ++i) {
            mbar_init(&bar.wfull[i], 1);
            mbar_init(&bar.wempty[i], 16);  // four chunks, four builder warps each
        }
        for (int i = 0; i < AP; ++i) {
            mbar_init(&bar.aready[i], 4);
            mbar_init(&bar.aempty[i], 1);
        }
        mbar_init(&bar.szfull, 1);
        mbar_init(&bar.accfull, n_iss);
        mbar_init(&bar.done, NBW);
        fence_barrier_init();
    }
    if (warp == 6) {  // allocates tensor memory and frees it at the end
        tmem_alloc(&bar.tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_holder;
    // programmatic dependent launch: this grid may start while the previous
    // launch of the stream finishes (its setup overlaps that launch's tail);
    // every global read and write follows the wait
    pdl_launch_dependents();
    pdl_wait();

    // the tile's scale and zero rows are contiguous in memory: one bulk copy
    // each (the last tile along N, when partial, is loaded by the builders)
    const bool full_tile = n0 + BR <= a.N;
    if (warp == 0) {
        // ---------------------------------------- packed codes (TMA)
        if (lane == 0) {
            if (full_tile) {
                const uint32_t tb = static_cast<uint32_t>(BR * a.G * 2);
                const uint64_t pol = policy_evict_last();  // every M tile reads them
                mbar_arrive_expect_tx(&bar.szfull, SYM ? tb : 2 * tb);
                bulk_g2s(s_t, a.s + static_cast<int64_t>(n0) * a.G, tb, &bar.szfull, pol);
                if (!SYM) bulk_g2s(z_t, a.z + static_cast<int64_t>(n0) * a.G, tb, &bar.szfull, pol);
            }
            tma_prefetch_desc(&tmW);
            const int nsc = (nch + 3) / 4;
            const int nissue = (a.inject & kInjectStallPipeline) ? 0 : nsc;
            int issued = 0;
            for (int sc = 0; sc < nissue; ++sc, ++issued) {
                const int ws = sc % WS;
                if (sc >= WS && !mbar_wait(&bar.wempty[ws], ((sc / WS) - 1) & 1, a.status)) break;
                mbar_arrive_expect_tx(&bar.wfull[ws], W_STAGE);
                // rows past N and codes past K/2 read as zeros
                tma_load_2d(smem + a.off_w + ws * W_STAGE, &tmW, (c0 / 4 + sc) * 128, n0, &bar.wfull[ws]);
            }
            for (int it = issued > WS ? issued - WS : 0; it < issued; ++it)
                mbar_wait(&bar.wfull[it % WS], (it / WS) & 1, nullptr);  // no copy in flight at exit
        }
    } else if (warp == 1) {
        // ------------------------------------------ X tiles (TMA)
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();  // every N tile of this M tile reads it
            tma_prefetch_desc(&tmX);
            const int nissue = (a.inject & kInjectStallPipeline) ? 0 : nch;
            int issued = 0;
            for (int c = 0; c < nissue; ++c, ++issued) {
                const int xs = c % xs_n;
                if (c >= xs_n && !mbar_wait(&bar.xempty[xs], ((c / xs_n) - 1) & 1, a.status)) break;
                mbar_arrive_expect_tx(&bar.xfull[xs], x_stage);
                // rows past M read as zeros
                tma_load_2d_hint(smem + xs * x_stage, &tmX, (c0 + c) * CK, m0, &bar.xfull[xs], pol);
            }
            for (int it = issued > xs_n ? issued - xs_n : 0; it < issued; ++it)
                mbar_wait(&bar.xfull[it % xs_n], (it / xs_n) & 1, nullptr);
        }
    } else if (warp >= ISS0 && warp < ISS0 + n_iss) {
        // ------------------------------------------------ MMA issuers
        const int j = warp - ISS0;
        const uint32_t d_acc = tmem + TM_ACC + static_cast<uint32_t>(j * nt);
        const uint32_t idesc = idesc_kind_f16(BR, nt, 0u);  // FP16 x FP16 -> FP32
        bool ok = !(a.inject & kInjectStallConsumers);
        for (int c = j; ok && c < nch; c += n_iss) {
            const int ap = c % AP, xs = c % xs_n;
            uint64_t *wbar = nullptr;
            uint32_t par = 0;
            if (lane == 0) {
                wbar = &bar.aready[ap];
                par = (c / AP) & 1;
            } else if (lane == 1) {
                wbar = &bar.xfull[xs];
                par = (c / xs_n) & 1;
            }
            if (!mbar_wait_lanes(wbar, par, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                const uint32_t b_addr = smem_u32(smem + xs * x_stage);
#pragma unroll
                for (int k = 0; k < CK / 16; ++k)
                    umma_f16_tmem_a_w(d_acc, tmem + TM_A + ap * 32 + 8 * k, smem_desc_sw128_kmajor(b_addr + 32 * k),
                                    idesc, (c != j) || (k != 0));
                umma_commit_w(&bar.xempty[xs]);
                umma_commit_w(&bar.aempty[ap]);
            }
            __syncwarp();
        }
        umma_commit_w(&bar.accfull);
        __syncwarp();
    } else if (warp == 6) {
        // tensor memory is freed only after every MMA has completed and the
        // epilogue has read the accumulators
        mbar_wait(&bar.accfull, 0, nullptr);
        mbar_wait(&bar.done, 0, a.status);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    } else if (warp >= BW0) {
        // ---------------- operand builders, then the epilogue
        for (int i = threadIdx.x - BW0 * 32; i < nt; i += NBW * 32)
            rs_t[i] = m0 + i < a.M ? a.rowscale[m0 + i] : 0.0f;  // read in the epilogue only
        if (!full_tile) {
            // the partial last tile along N: rows past N get zero scales
            const int bt = threadIdx.x - BW0 * 32;  // 0 .. NBW * 32 - 1
            for (int e = bt; e < BR * a.G; e += NBW * 32) {
                const int rr = e / a.G;
                const bool in = n0 + rr < a.N;
                const int64_t at = static_cast<int64_t>(n0) * a.G + e;
                s_t[e] = in ? a.s[at] : static_cast<uint16_t>(0);
                if (!SYM) z_t[e] = in ? a.z[at] : static_cast<uint16_t>(0);
            }
            named_bar_sync(1, NBW * 32);
            if (bt == 0) mbar_arrive(&bar.szfull);
        }

        const int q = warp & 3;
        const int grp = (warp - BW0) >> 2;  // chunks grp, grp + BG, ...
        const int r = q * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        bool ok = mbar_wait(&bar.szfull, 0, a.status);
        for (int c = grp; ok && c < nch; c += BG) {
            const int sc = c >> 2, ws = sc % WS, ap = c % AP;
            uint64_t *wbar = nullptr;
            uint32_t wpar = 0;
            if (lane == 0) {
                wbar = &bar.wfull[ws];
                wpar = (sc / WS) & 1;
            } else if (lane == 1 && c >= AP) {
                wbar = &bar.aempty[ap];
                wpar = ((c - AP) / AP) & 1;
            }
            if (!mbar_wait_lanes(wbar, wpar, a.status)) {
                ok = false;
                break;
            }
            // the group's scale and zero point, as binary16 pairs
            const int g = (c0 + c) >> 1;  // two chunks per group
            const uint32_t sh = s_t[r * a.G + g];
            const uint32_t zh = SYM ? 0x4800u : static_cast<uint32_t>(z_t[r * a.G + g]);  // 8.0 when symmetric
            const uint32_t s2 = sh | (sh << 16);
            const uint32_t z2 = zh | (zh << 16);
            // this row's 32 code bytes of the chunk: 16-byte chunks
            // 2 (c mod 4) and 2 (c mod 4) + 1 of the swizzled 128-byte row
            const unsigned char *wrow = smem + a.off_w + ws * W_STAGE + r * 128;
            const int j0 = 2 * (c & 3);
            const uint4 v0 = *reinterpret_cast<const uint4 *>(wrow + ((j0 ^ (r & 7)) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4 *>(wrow + (((j0 + 1) ^ (r & 7)) << 4));
            const uint32_t wds[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            uint32_t cols[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t w = wds[u];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // codes i and i + 4 of the word: q + 1024 in binary16, exact
                    const uint32_t qm = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
                    cols[4 * u + i] = hmul2(hsub2(hsub2(qm, 0x64006400u), z2), s2);
                }
            }
            tmem_st_32x32b_x32(tmem + t_lane + TM_A + ap * 32, cols);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar.aready[ap]);
                mbar_arrive(&bar.wempty[ws]);
            }
        }
        // epilogue: group g stores the 16-column pieces p = g, g + BG, ... of
        // the tile's token rows, each the sum of the issuers' accumulators
        named_bar_sync(2, NBW * 32);  // the row scales are in shared memory
        ok = ok && mbar_wait_lanes(lane == 0 ? &bar.accfull : nullptr, 0, a.status);
        const int rows_m = min(nt, a.M - m0);
        // With y_tma the tile goes to shared memory as [token][128 rows] BF16
        // -- into the X ring, idle once every MMA has completed -- and leaves
        // by one TMA store (rows past M and N are not written).
        uint16_t *ytile = reinterpret_cast<uint16_t *>(smem);
        if (ok) {
            tc_fence_after();
            const bool nok = n0 + r < a.N;
            uint16_t *yrow = a.Y + n0 + r;
            for (int p = grp; 16 * p < rows_m; p += BG) {
                float acc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
                for (int jj = 0; jj < n_iss; ++jj) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tmem + t_lane + TM_ACC + static_cast<uint32_t>(jj * nt + 16 * p), v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(v[i]);
                }
                if (partial) {
                    // a K-split tile: binary32 sums [m][r], finished (summed,
                    // scaled, rounded) by the reduction launch
                    float *dst = a.part + static_cast<int64_t>(part_id) * nt * BR + r;
#pragma unroll
                    for (int i = 0; i < 16; ++i) dst[static_cast<int64_t>(16 * p + i) * BR] = acc[i];
                } else if (y_tma) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        ytile[(16 * p + i) * BR + r] = f32_to_bf16_bits(acc[i] * rs_t[16 * p + i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = m0 + 16 * p + i;
                        if (16 * p + i < rows_m && nok)
                            yrow[static_cast<int64_t>(m) * a.N] = f32_to_bf16_bits(acc[i] * rs_t[16 * p + i]);
                    }
                }
            }
        }
        if (y_tma) {
            // every builder's part written (generic proxy), then one store
            fence_proxy_async_smem();
            named_bar_sync(3, NBW * 32);
            if (ok && threadIdx.x == BW0 * 32) {
                tma_store_2d(&tmY, n0, m0, ytile);
                bulk_commit_group();
                bulk_wait_read_all();  // shared memory is read before the CTA ends
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.done);
    }
}

// The K-split tiles' outputs: Y[m0 + m, n0 + r] = RNE_bf16(rowscale[m0 + m]
// x sum over the splits of part[x][y][m][r]), splits summed in order from
// zero.  One CTA per (tile x, 32 token rows); thread t takes weight rows
// 4 (t mod 32) .. + 3 (one 16-byte load per split) of token rows
// 8 k + t / 32, k = 0..3, so that many loads are in flight per thread (the
// parts are in L2, just written).
constexpr int RED_THREADS = 256;
constexpr int RED_ROWS = 32;  // token rows per CTA
__global__ void __launch_bounds__(RED_THREADS) f16_split_reduce_kernel(const float *__restrict__ part,
                                                                       const float *__restrict__ rowscale,
                                                                       uint16_t *Y, int M, int N, int nt, int ntn,
                                                                       int tile0, int nsplit) {
    pdl_launch_dependents();
    pdl_wait();  // the partial sums and the row scales follow the stream order
    const int x = blockIdx.x;
    const int tile = tile0 + x;
    const int n0 = (tile % ntn) * BR, m0 = (tile / ntn) * nt;
    const int r = 4 * (threadIdx.x & 31);
    const int64_t split_stride = static_cast<int64_t>(nt) * (BR / 4);  // float4 units
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float4 *base = reinterpret_cast<const float4 *>(part) + static_cast<int64_t>(x) * nsplit * split_stride;
    int mk[4];
    bool in[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        mk[k] = blockIdx.y * RED_ROWS + 8 * k + (threadIdx.x >> 5);
        in[k] = mk[k] < nt && m0 + mk[k] < M;
    }
#pragma unroll 2
    for (int y = 0; y < nsplit; ++y) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (!in[k]) continue;
            const float4 v = base[y * split_stride + (static_cast<int64_t>(mk[k]) * BR + r) / 4];
            acc[k].x += v.x;
            acc[k].y += v.y;
            acc[k].z += v.z;
            acc[k].w += v.w;
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (!in[k]) continue;
        const float rs = rowscale[m0 + mk[k]];
        uint16_t *dst = Y + static_cast<int64_t>(m0 + mk[k]) * N + n0 + r;
        const float v[4] = {acc[k].x, acc[k].y, acc[k].z, acc[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (n0 + r + e < N) dst[e] = f32_to_bf16_bits(v[e] * rs);
    }
}

// A memory pool per device for the pre-pass output (stream-ordered, kept
// reserved between calls).
struct PrepassPool {
    std::mutex mu;
    cudaMemPool_t pool[64] = {};
};
PrepassPool g_pool;

cudaError_t prepass_pool(int device, cudaMemPool_t &out) {
    std::lock_guard<std::mutex> lk(g_pool.mu);
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (!g_pool.pool[device]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = device;
        cudaMemPool_t p;
        if (cudaError_t e = cudaMemPoolCreate(&p, &props)) return e;
        uint64_t keep = ~0ull;
        if (cudaError_t e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep)) {
            cudaMemPoolDestroy(p);
            return e;
        }
        g_pool.pool[device] = p;
    }
    out = g_pool.pool[device];
    return cudaSuccess;
}

// Shared-memory layout: [X ring][packed-code ring][scale (and zero) tiles][barriers].
struct F16Layout {
    int nt, xs_n, off_w, off_sz, off_bar, bytes;
};

// The X ring takes what the packed-code ring, the scale/zero tiles and the
// barriers leave (it is what covers the L2 round trip of the X tiles).
F16Layout f16_layout(int64_t M, int64_t K, bool sym) {
    F16Layout l;
    l.nt = M >= NT_MAX ? NT_MAX : static_cast<int>((M + 15) / 16) * 16;
    const int n_iss = l.nt <= 64 ? MAX_ISS : (l.nt <= 128 ? 2 : 1);
    const int G = static_cast<int>(K / GK);
    const int fixed = 1024 + WS * W_STAGE + (sym ? 1 : 2) * BR * G * 2 + NT_MAX * 4 + static_cast<int>(sizeof(Barriers));
    int xs_n = (SMEM_BUDGET - fixed) / (l.nt * 128);
    xs_n = xs_n < XS_MAX ? xs_n : XS_MAX;
    xs_n -= xs_n % n_iss;  // a multiple of the issuer count (n_iss = 4 only when nt <= 64: room for 8)
    l.xs_n = xs_n;
    l.off_w = xs_n * l.nt * 128;
    l.off_sz = l.off_w + WS * W_STAGE;
    l.off_bar = l.off_sz + (sym ? 1 : 2) * BR * G * 2 + NT_MAX * 4;  // 16-byte aligned (256 G per tile)
    l.bytes = 1024 + l.off_bar + static_cast<int>(sizeof(Barriers));
    // at least half of an SM's shared memory: one CTA per SM, so that no
    // CTA waits in tcgen05.alloc for another's 512 columns
    l.bytes = l.bytes > 116 * 1024 ? l.bytes : 116 * 1024;
    return l;
}

}  // namespace

int gemm_int4_f16_smem(int64_t M, int64_t K, bool sym) { return f16_layout(M, K, sym).bytes; }

cudaError_t launch_gemm_int4_f16(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const uint16_t *z,
                                 uint16_t *Y, int64_t M, int64_t N, int64_t K, cudaStream_t st, unsigned int *status,
                                 const DeviceInfo &dev) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    if (K / 8 > static_cast<int64_t>(PRE_BLOCKS) * PRE_THREADS) return cudaErrorNotSupported;  // the pre-pass's reach
    const bool sym = z == nullptr;
    const F16Layout lay = f16_layout(M, K, sym);
    const int nt = lay.nt;
    const int smem = lay.bytes;
    if (smem > dev.max_smem_optin || lay.xs_n < 2) return cudaErrorNotSupported;
    const int64_t ntn = (N + BR - 1) / BR, ntm = (M + nt - 1) / nt;
    if (ntn * ntm > 0x7FFFFFFFll || M > 0x7FFFFFFFll) return cudaErrorInvalidValue;

    // Tiles past the last full wave of CTAs (one CTA per SM): when they fill
    // at most half a wave, each is split along K into nsplit parts of whole
    // packed-code stages (at least two of them).  The parts are the launch's
    // last CTAs, so they take the SMs as the last whole tiles finish, and a
    // reduction launch finishes them from their binary32 partial sums.  With
    // 960 tiles on 152 SMs (M = 2048, N = 15360) the last 48 tiles would
    // otherwise make a seventh wave of whole tiles on a third of the SMs.
    const int64_t tiles = ntn * ntm;
    const int nch_all = static_cast<int>(K / CK);
    int64_t tiles_full = tiles, tiles_split = 0;
    int cps = nch_all, nsplit = 1;
    if (K % 256 == 0 && tiles > dev.num_sms) {
        const int64_t rest = tiles % dev.num_sms;
        if (rest > 0 && 2 * rest <= dev.num_sms) {
            int parts = static_cast<int>(dev.num_sms / rest);
            if (parts > nch_all / 8) parts = nch_all / 8;
            if (parts >= 2) {
                cps = ((nch_all + parts - 1) / parts + 3) / 4 * 4;
                nsplit = (nch_all + cps - 1) / cps;
                tiles_split = rest;
                tiles_full = tiles - rest;
            }
        }
    }

    // 1. pre-pass into stream-ordered scratch: X16 [M, K] binary16, the row
    // scales, and the K-split tiles' partial sums
    cudaMemPool_t pool;
    if (cudaError_t e = prepass_pool(dev.device, pool)) return e;
    const size_t xh_bytes = (static_cast<size_t>(M) * static_cast<size_t>(K) * 2 + 255) & ~size_t(255);
    const size_t rs_bytes = (static_cast<size_t>(M) * 4 + 255) & ~size_t(255);
    const size_t part_bytes = static_cast<size_t>(tiles_split) * nsplit * nt * BR * 4;
    void *scr = nullptr;
    if (cudaError_t e = cudaMallocFromPoolAsync(&scr, xh_bytes + rs_bytes + part_bytes, pool, st)) return e;
    uint16_t *xh = static_cast<uint16_t *>(scr);
    float *rowscale = reinterpret_cast<float *>(static_cast<unsigned char *>(scr) + xh_bytes);
    float *part = tiles_split ? reinterpret_cast<float *>(static_cast<unsigned char *>(scr) + xh_bytes + rs_bytes)
                              : nullptr;
    // the pre-pass and the GEMM are launched with programmatic stream
    // serialisation: each may start while the previous launch finishes and
    // waits for it (griddepcontrol.wait) before touching global memory
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaError_t err;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(M));
        cfg.blockDim = dim3(PRE_THREADS);
        cfg.stream = st;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        const int64_t per_thread = (K / 8 + PRE_THREADS - 1) / PRE_THREADS;
        err = per_thread <= 2   ? cudaLaunchKernelEx(&cfg, x16_prepass_kernel<2>, X, static_cast<int>(K), xh, rowscale)
              : per_thread <= 4 ? cudaLaunchKernelEx(&cfg, x16_prepass_kernel<4>, X, static_cast<int>(K), xh, rowscale)
                                : cudaLaunchKernelEx(&cfg, x16_prepass_kernel<8>, X, static_cast<int>(K), xh, rowscale);
    }

    // 2. the GEMM
    CUtensorMap tmW, tmX, tmY;
    memset(&tmY, 0, sizeof(tmY));
    const int y_tma = N % 8 == 0 ? 1 : 0;
    if (err == cudaSuccess) {
        // packed codes as bytes [N, K/2]: box 128 bytes (256 codes) x 128 rows, 128-byte swizzle
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
        const cuuint32_t box[2] = {128, BR};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(qw), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            err = cudaErrorInvalidValue;
    }
    if (err == cudaSuccess) {
        // X16 [M, K]: box 64 (128 bytes) x NT rows, 128-byte swizzle
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(nt)};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xh, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            err = cudaErrorInvalidValue;
    }
    if (err == cudaSuccess && y_tma) {
        // Y [M, N] BF16: box 128 columns (256 bytes) x NT rows, no swizzle
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
        const cuuint32_t box[2] = {BR, static_cast<cuuint32_t>(nt)};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Y, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            err = cudaErrorInvalidValue;
    }
    if (err == cudaSuccess) {
        GemmF16Args a;
        a.s = s;
        a.z = z;
        a.rowscale = rowscale;
        a.Y = Y;
        a.status = status;
        a.M = static_cast<int>(M);
        a.N = static_cast<int>(N);
        a.K = static_cast<int>(K);
        a.G = static_cast<int>(K / GK);
        a.nt = nt;
        a.ntn = static_cast<int>(ntn);
        a.xs_n = lay.xs_n;
        a.off_w = lay.off_w;
        a.off_sz = lay.off_sz;
        a.off_bar = lay.off_bar;
        a.y_tma = y_tma;
        a.inject = dev.inject;
        a.tiles_full = static_cast<int>(tiles_full);
        a.nsplit = nsplit;
        a.cps = cps;
        a.part = part;
        const void *kern = sym ? reinterpret_cast<const void *>(gemm_int4_f16_kernel<true>)
                               : reinterpret_cast<const void *>(gemm_int4_f16_kernel<false>);
        static SmemLimit limit[2];  // one per kernel instance
        err = limit[sym ? 1 : 0].ensure(kern, dev.device, smem);
        if (err == cudaSuccess) {
            // whole tiles first, the K-split parts last: they fill the SMs as
            // the last whole tiles finish
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(tiles_full + tiles_split * nsplit));
            cfg.blockDim = dim3(THREADS);
            cfg.dynamicSmemBytes = static_cast<size_t>(smem);
            cfg.stream = st;
            cfg.attrs = pdl;
            cfg.numAttrs = 1;
            err = sym ? cudaLaunchKernelEx(&cfg, gemm_int4_f16_kernel<true>, tmW, tmX, tmY, a)
                      : cudaLaunchKernelEx(&cfg, gemm_int4_f16_kernel<false>, tmW, tmX, tmY, a);
        }
        if (err == cudaSuccess && tiles_split) {
            // the K-split tiles' outputs from their partial sums
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(tiles_split), static_cast<unsigned>((nt + RED_ROWS - 1) / RED_ROWS));
            cfg.blockDim = dim3(RED_THREADS);
            cfg.stream = st;
            cfg.attrs = pdl;
            cfg.numAttrs = 1;
            err = cudaLaunchKernelEx(&cfg, f16_split_reduce_kernel, static_cast<const float *>(part),
                                     static_cast<const float *>(rowscale), Y, static_cast<int>(M), static_cast<int>(N),
                                     nt, static_cast<int>(ntn), static_cast<int>(tiles_full), nsplit);
        }
    }
    // the scratch returns to the pool once the work queued on the stream is done
    cudaError_t fe = cudaFreeAsync(scr, st);
    return err != cudaSuccess ? err : fe;
}

}  // namespace w4
