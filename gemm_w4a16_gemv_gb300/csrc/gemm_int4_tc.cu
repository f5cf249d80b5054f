// Prefill GEMM with INT4 group-128 weights on the tcgen05 tensor cores:
//   Y[m, n] = sum_k X[m, k] * (q[n, k] - z[n, k/128]) * s[n, k/128]
// ("Lab 5: Gemma4 end-to-end inference optimisation": prefill (M > 1) went
// through a Triton dequantiser writing BF16 weights and a cuBLAS GEMM; here the
// dequantised weight tile never leaves the SM, so HBM sees only packed codes).
//
// The dequantisation is split into an exact part that feeds the tensor cores
// and an affine part applied per group to the accumulator.  With
// z_i = clamp(rint(z), 0, 15) and the residual z_r = z - z_i (zero whenever
// z is an integer code, as GPTQ zero points are):
//   sum_{k in g} X[m,k] (q - z) s = s * A_g[n,m] - s * z_r * S_g[m]
//   A_g[n,m] = sum_{k in g} (q[n,k] - z_i) * X[m,k]    (BF16 x BF16 MMA)
//   S_g[m]   = sum_{k in g} X[m,k]                      (same MMA: rows of ones)
// q - z_i is an integer in [-15, 15], so the weight operand is an exact BF16
// number and X enters as loaded; every product is exact and all sums are
// binary32.  When every z_r of a warp's rows is zero for a group (the
// common case) the epilogue is one multiply-add per element; otherwise it
// also folds in S_g.
//
// Operand placement.  The weights are the MMA's A operand and live in tensor
// memory: in each 32-lane quarter of the 128 TMEM lanes, lanes 0-27 hold 28
// weight rows and lanes 28-31 BF16 ones, whose accumulator rows give S_g (so
// an epilogue warp that needs S_g finds it in its own lane 28 and broadcasts
// it with a shuffle).  The activation tile is the B operand (N = 128 rows m
// of X) in shared memory, loaded by TMA.  So shared memory carries only the X
// tiles (written by TMA, read by the MMA) and the packed codes; the
// dequantised weights go straight from registers to TMEM (tcgen05.st).
//
// Every hand-off is per group (128 K, two TMA boxes of 64): an mbarrier wait
// costs about 200 SM cycles of latency on this part even when the phase has
// already completed, so each role waits once per group, not per MMA step.
//
// One CTA computes a tile of 112 output columns n x 128 rows m; each CTA
// loads its own X tiles (from L2 after the first CTA that needs them):
//  * warp 0: the tile's scale and zero rows (16-byte cp.async chunks); then,
//    from one lane, per group its X rows (two TMA boxes, 128-byte swizzle);
//  * warp 2 (one lane): every two groups the packed codes of the tile's rows,
//    128 bytes each (TMA), on a ring of its own;
//  * warps 8-11 (even groups) and 16-19 (odd groups), TMEM lane quarters
//    0-3: per group, thread (q, i) turns the 128 codes of weight row 28 q + i
//    into 64 columns of BF16 pairs q - z_i (byte permutes and one BF16 pair
//    subtraction) and stores them into the group's TMEM operand stage; lanes
//    28-31 store ones;
//  * warps 1 and 3 (one lane each) issue the MMAs of the even and the odd
//    groups, so that one warp's barrier checks overlap the other's issue and
//    the tensor pipe sees a steady stream: per group wait for the operand
//    stage (one of four), the X tile and a free accumulator (one of two),
//    issue 8 x tcgen05.mma (M=128, N=128, K=16, A from TMEM) and commit
//    three times: to the X stage's barrier, to the operand stage's and to
//    the accumulator's;
//  * warps 4-7 and 12-15: per group load the accumulator (warp w: TMEM lanes
//    32 (w mod 4) .. +31, one half of the 128 columns) into registers,
//    release it at once and fold y += s A_g (- s z_r S_g) into registers;
//    at the end round to BF16 and store Y.
// Every wait is bounded; on timeout the status word is set, each role still
// performs the arrivals the others wait for, and TMEM is released only after
// every MMA issued has completed.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace w4 {
namespace {

constexpr int BNW = 112;              // weight rows per tile: 28 in each TMEM lane quarter
constexpr int RQ = 28;                // weight rows per lane quarter (lanes 28-31: ones)
constexpr int BM = 128;               // X rows per tile at most (the MMA's N): M rounded up to 16 below 128
constexpr int BK = 64;                // one TMA box of X (128 bytes of BF16 per row)
constexpr int GK = 128;               // K per group = per hand-off
constexpr int MAX_XP = 5;             // X ring depth in groups (runtime, from shared memory)
constexpr int WS = 3;                 // packed-code ring (each load: two groups)
constexpr int AP = 4;                 // TMEM operand stages (64 columns each)
constexpr int DB = 2;                 // TMEM accumulators (128 columns each)
constexpr int W_BYTES = BNW * 128;    // 14 KB packed codes, two groups
constexpr int THREADS = 640;          // 20 warps, five warpgroups
constexpr int PREP_WARPS = 8;         // warps 8-11 (even groups) and 16-19 (odd groups)
constexpr int PREP_PER_GROUP = 4;     // one builder warp per lane quarter builds a group
constexpr int EPI_WARPS = 8;          // warps 4-7, 12-15
constexpr uint32_t TMEM_COLS = 512;
// Registers per thread after the per-warpgroup split (setmaxnreg): the light
// warps and the builders release down to theirs, the epilogue grows to its
// own, so the launch count must lie between them (checked by the launcher).
constexpr uint32_t kRegLight = 32;    // warps 0-3: producers and MMA issuers
constexpr uint32_t kRegBuild = 80;    // warps 8-11, 16-19: operand builders
constexpr uint32_t kRegEpi = 144;     // warps 4-7, 12-15: epilogue
constexpr int kRegSplit = 128 * static_cast<int>(kRegLight + 2 * kRegEpi + 2 * kRegBuild);
// Suspend-time hints (ns) of the waits' polls, per role (0: plain polls).
constexpr uint32_t kHintProd = 0;     // X and packed-code producers
constexpr uint32_t kHintMma = 0;      // MMA issuers
constexpr uint32_t kHintBuild = 0;    // operand builders
constexpr uint32_t kHintEpi = 0;      // epilogue
constexpr uint32_t TM_A = DB * 128;   // operand stages after the accumulators
constexpr uint32_t ONES = 0x3F803F80u;  // two BF16 1.0
// layout: [X ring][W ring][s tile][z tile][barriers]
constexpr int OFF_X = 0;
constexpr int MAX_K = 16384;

struct GemmArgs {
    const uint16_t *s;
    const uint16_t *z;
    uint16_t *Y;
    unsigned int *status;
    int M, N, K, G;
    int sz_bytes;  // bytes of one staged scale (or zero) tile, 16-aligned
    int xp;        // X ring depth in groups
    int off_w, off_sz;
    unsigned int inject;  // test-only injection flags (0 normally); kept after
                          // the hot fields: inserting it earlier shifted them
                          // and measurably slowed the kernel
    int bm;               // X rows per tile: min(128, M rounded up to 16)
};

struct Barriers {
    uint64_t xfull[MAX_XP];   // a group's X tile landed (TMA tx bytes)
    uint64_t xempty[MAX_XP];  // MMAs done with the group
    uint64_t wfull[WS];       // packed codes landed (TMA tx bytes)
    uint64_t wempty[WS];      // packed codes read (operand builders)
    uint64_t aready[AP];      // TMEM operand stage written (operand builders)
    uint64_t aempty[AP];      // MMAs done with the operand stage (commit, local)
    uint64_t accfull[DB];     // group accumulator complete (commit)
    uint64_t accempty[DB];    // group accumulator read (epilogue warps)
    uint64_t szfull;          // scale/zero tiles landed
    uint64_t done;            // epilogue and operand builders finished with TMEM
    uint64_t drained;         // every MMA of both issuing warps completed (commits)
    uint32_t tmem_holder;
};

// SYM: symmetric INT4 (no zero points, z = 8), its own instance so that the
// asymmetric one carries no test for it.
template <bool SYM>
__global__ void __launch_bounds__(THREADS, 1)
gemm_int4_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const GemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    // X tiles and packed-code tiles use the 128-byte swizzle: 1024-byte alignment
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint16_t *s_tile = reinterpret_cast<const uint16_t *>(smem + a.off_sz);
    const uint16_t *z_tile = reinterpret_cast<const uint16_t *>(smem + a.off_sz + a.sz_bytes);
    Barriers &bar = *reinterpret_cast<Barriers *>(smem + a.off_sz + 2 * a.sz_bytes);
    const int XP = a.xp;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BNW;
    const int bm = a.bm;
    const int x_stage = 2 * bm * BK * 2;  // a group's X: [2][bm rows][128 bytes]
    const int m0 = blockIdx.y * bm;
    const int ngroups = a.G;
    const int rows_n = max(0, min(BNW, a.N - n0));  // weight rows of this tile

    if (threadIdx.x == 0) {
        for (int i = 0; i < XP; ++i) {
            mbar_init(&bar.xfull[i], 1);
            mbar_init(&bar.xempty[i], 1);
        }
        for (int i = 0; i < WS; ++i) {
            mbar_init(&bar.wfull[i], 1);
            mbar_init(&bar.wempty[i], PREP_WARPS);
        }
        for (int i = 0; i < AP; ++i) {
            mbar_init(&bar.aready[i], PREP_PER_GROUP);
            mbar_init(&bar.aempty[i], 1);
        }
        for (int i = 0; i < DB; ++i) {
            mbar_init(&bar.accfull[i], 1);
            mbar_init(&bar.accempty[i], EPI_WARPS);
        }
        mbar_init(&bar.szfull, 32);  // the 32 lanes of the producer warp (cp.async arrivals)
        mbar_init(&bar.done, EPI_WARPS + PREP_WARPS);
        mbar_init(&bar.drained, 2);
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
    // programmatic dependent launch: this grid may start while the previous
    // launch of the stream finishes (its setup overlaps that launch's tail);
    // every global read and write follows the wait
    pdl_launch_dependents();
    pdl_wait();

    // Registers per warpgroup, set at the top of each role: the producers and
    // MMA issuers (warps 0-3) need few; each epilogue thread (warps 4-7,
    // 12-15) holds 64 running sums and a 64-column accumulator slice; the
    // operand builders (8-11, 16-19) a group's 16 code words and 32 columns.
    // 128 threads x (32 + 144 + 80 + 144 + 80) = kRegSplit registers.  The
    // launcher checks that the block is launched with at least that many (a
    // shortfall would leave setmaxnreg.inc waiting) and with a per-thread
    // count between the released and the acquired ones (an increase below,
    // or a decrease above, the current count is not a valid instruction).
    if (warp == 0) {
        reg_release<kRegLight>();
        // ------------------------------------------------------ TMA producer
        // the whole warp waits (one lane per barrier); lane 0 issues.  X is
        // kept in L2 (evict-last): every N tile reads it, and the streamed
        // packed codes (evict-first) must not push it out.
        const uint64_t pol = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        if (lane == 0) {
            tma_prefetch_desc(&tmW);
            tma_prefetch_desc(&tmX);
        }
        {
            // the tile's scale (and zero) rows: one contiguous byte range
            // starting 16-byte aligned (n0 is a multiple of 112), copied in
            // 16-byte chunks by the warp's lanes; a chunk past the tensor's
            // end (any N) reads only the bytes before it and zero-fills the rest
            const uint64_t b0 = static_cast<uint64_t>(n0) * a.G * 2;
            const uint64_t b1 = b0 + static_cast<uint64_t>(rows_n) * a.G * 2;
            const uint64_t total = static_cast<uint64_t>(a.N) * a.G * 2;
            const unsigned char *gs = reinterpret_cast<const unsigned char *>(a.s);
            const unsigned char *gz = reinterpret_cast<const unsigned char *>(a.z);
            for (uint64_t o = b0 + 16 * static_cast<uint64_t>(lane); o < b1; o += 16 * 32) {
                const uint32_t n = total - o < 16 ? static_cast<uint32_t>(total - o) : 16u;
                cp_async_16_zfill(smem + a.off_sz + (o - b0), gs + o, n);
                if (!SYM) cp_async_16_zfill(smem + a.off_sz + a.sz_bytes + (o - b0), gz + o, n);
            }
            cp_async_arrive_noinc(&bar.szfull);  // counts once per lane
        }
        int xs = 0, xph = 0;  // X stage and its phase
        // test-only injection: no X stage is ever issued, so the waits on it
        // run out and the launch ends with the timeout status
        const int xgroups = (a.inject & kInjectStallPipeline) ? 0 : ngroups;
        int issued = 0;
        for (int g = 0; g < xgroups; ++g, ++issued) {
            if (g >= XP && !mbar_wait<kHintProd>(&bar.xempty[xs], xph ^ 1, a.status)) break;
            if (lane == 0) {
                // the group's two 64-K halves in one copy: [2][bm rows][128 bytes]
                mbar_arrive_expect_tx(&bar.xfull[xs], 2 * bm * BK * 2);
                tma_load_3d_hint(smem + OFF_X + xs * x_stage, &tmX, 0, m0, 2 * g, &bar.xfull[xs], pol_x);
            }
            __syncwarp();
            if (++xs == XP) {
                xs = 0;
                xph ^= 1;
            }
        }
        // No copy of this CTA may still be landing when it exits: wait
        // (bounded, whatever the status word says) for the tiles issued and
        // not known to be consumed, and for the scale/zero copies.
        for (int it = issued > XP ? issued - XP : 0; it < issued; ++it)
            mbar_wait(&bar.xfull[it % XP], (it / XP) & 1, nullptr);
        mbar_wait(&bar.szfull, 0, nullptr);
    } else if (warp == 2) {
        reg_release<kRegLight>();
        // ---------------------------------------- packed-code TMA producer
        // its own ring, so the codes (from HBM) are requested as early as the
        // ring allows, independently of the X ring's pace; streamed with the
        // evict-first policy
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const int nwb = (ngroups + 1) / 2;
            int issued = 0;
            for (int wb = 0; wb < nwb; ++wb, ++issued) {
                const int ws = wb % WS;
                if (wb >= WS && !mbar_wait<kHintProd>(&bar.wempty[ws], ((wb / WS) - 1) & 1, a.status)) break;
                mbar_arrive_expect_tx(&bar.wfull[ws], W_BYTES);
                // rows past N (last and padding tiles) read as zeros
                tma_load_2d_hint(smem + a.off_w + ws * W_BYTES, &tmW, wb * 128, n0, &bar.wfull[ws], pol_w);
            }
            // as for the X tiles: no copy in flight when the CTA exits
            for (int it = issued > WS ? issued - WS : 0; it < issued; ++it)
                mbar_wait(&bar.wfull[it % WS], (it / WS) & 1, nullptr);
        }
    } else if (warp == 1 || warp == 3) {
        reg_release<kRegLight>();
        // ------------------------------------------------------ MMA issuers
        // warp 1 takes the even groups, warp 3 the odd ones.  The whole warp
        // waits for its group's three conditions at once (one lane per
        // barrier); lane 0 issues.  Ring positions advance two groups per
        // step (XP >= 3, DB = 2, AP = 4: at most one wrap each).
        //
        // A parity wait passes at once if its barrier is still in the phase
        // before the awaited one, so no wait may run two phases ahead.  The
        // accumulators (DB = 2) and operand stages (AP = 4) belong to one
        // issuer each; an X stage's previous group g - XP belongs to the same
        // issuer when XP is even, and when XP >= DB + 2 it was released (its
        // MMAs done) before this issuer's accumulator wait for group g - 2
        // ended.  With XP = 3 (the largest K) the X stage is awaited only
        // after the accumulator, in a second round.
        const uint32_t idesc = idesc_kind_f16(128, bm, 1u);  // BF16, M = 128 lanes, N = bm rows of X
        const bool x_second = (XP & 1) && XP < DB + 2;
        // test-only injection: the issuers take nothing, so the producers'
        // waits for free stages run out with their copies issued
        const int g0 = warp == 1 ? 0 : 1;
        bool ok = !(a.inject & kInjectStallConsumers);
        int xs = g0, xph = 0, db = g0, dph = 0, ap = g0, aph = 0;
        for (int g = g0; ok && g < ngroups; g += 2) {
            uint64_t *wbar = nullptr;
            uint32_t par = 0;
            if (lane == 0) {
                wbar = &bar.aready[ap];
                par = aph;
            } else if (lane == 1 && !x_second) {
                wbar = &bar.xfull[xs];
                par = xph;
            } else if (lane == 2 && g >= DB) {
                wbar = &bar.accempty[db];
                par = dph ^ 1;
            }
            if (!mbar_wait_lanes<kHintMma>(wbar, par, a.status) ||
                (x_second && !mbar_wait_lanes<kHintMma>(lane == 1 ? &bar.xfull[xs] : nullptr, xph, a.status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                const uint32_t t_acc = tmem + db * 128;
                const uint32_t a_t = tmem + TM_A + ap * 64;
                const uint32_t b_addr = smem_u32(smem + OFF_X + xs * x_stage);
#pragma unroll
                for (int k = 0; k < GK / 16; ++k)
                    umma_f16_tmem_a_w(t_acc, a_t + 8 * k,
                                      smem_desc_sw128_kmajor(b_addr + (k >> 2) * (bm * BK * 2) + 32 * (k & 3)), idesc,
                                      k != 0);
                umma_commit_w(&bar.xempty[xs]);
                umma_commit_w(&bar.aempty[ap]);
                umma_commit_w(&bar.accfull[db]);
            }
            __syncwarp();
            xs += 2;
            if (xs >= XP) {
                xs -= XP;
                xph ^= 1;
            }
            db += 2;
            if (db >= DB) {
                db -= DB;
                dph ^= 1;
            }
            ap += 2;
            if (ap >= AP) {
                ap -= AP;
                aph ^= 1;
            }
        }
        // Only after a timeout: one more commit so that the epilogue's wait
        // for this warp's group also ends once the MMAs already issued have
        // completed.
        if (!ok) umma_commit_w(&bar.accfull[db]);
        // `drained` fires once every MMA of both warps has completed
        umma_commit_w(&bar.drained);
        __syncwarp();
        if (warp == 1) {
            // MMAs always complete, so this wait ignores the status word: TMEM
            // is never released under an MMA still in flight
            mbar_wait<kHintMma>(&bar.drained, 0, nullptr);
            mbar_wait<kHintMma>(&bar.done, 0, a.status);
            __syncwarp();
            tc_fence_after();
            tmem_dealloc(tmem, TMEM_COLS);
        }
    } else if ((warp >= 8 && warp < 12) || warp >= 16) {
        // ---------------------------------------------- TMEM operand builders
        // two warps per lane quarter: warps 8-11 build the even groups, 16-19
        // the odd ones, so each has two group periods for its chain of
        // waits, loads, conversion and stores (one warp per group is bound by
        // that chain's latency, not by issue)
        reg_release<kRegBuild>();
        const int q = warp & 3;
        const int gpar = warp >= 16 ? 1 : 0;
        const int n = q * RQ + lane;  // weight row of this thread (lanes < 28)
        const bool wrow_ok = lane < RQ;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        const bool zrow = !SYM && wrow_ok && n < rows_n;  // rows with loaded zero points
        // warp-uniform waits throughout (one lane per barrier)
        const bool okb = mbar_wait_lanes<kHintBuild>(lane == 0 ? &bar.szfull : nullptr, 0, a.status);
        // Parity waits stay in phase: each operand stage belongs to one group
        // parity (AP even), and both parities meet every packed-code box in
        // order (one group of each box per parity).
        for (int g = gpar; okb && g < ngroups; g += 2) {
            const int ap = g % AP;
            const int wb = g >> 1, ws = wb % WS, half = g & 1;
            // lane 0: the packed codes; lane 1: operand stage ap is free once
            // the MMAs of group g - AP are done (their commit to the stage's
            // own barrier)
            uint64_t *wbar = nullptr;
            uint32_t par = 0;
            if (lane == 0) {
                wbar = &bar.wfull[ws];
                par = (wb / WS) & 1;
            } else if (lane == 1 && g >= AP) {
                wbar = &bar.aempty[ap];
                par = ((g - AP) / AP) & 1;
            }
            if (!mbar_wait_lanes<kHintBuild>(wbar, par, a.status)) break;
            // The group's 64 code bytes of row n (16-byte chunks 4 half + 0..3
            // of the swizzled packed stage, chunk j at j ^ (n mod 8)) are
            // loaded together: a shared-memory load waits several hundred
            // cycles here (the TMA and the MMAs share the port), so both
            // halves' loads must be in flight at once.
            uint32_t wds[16];
            if (wrow_ok) {
                const unsigned char *wrow = smem + a.off_w + ws * W_BYTES + n * 128;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const uint4 p = *reinterpret_cast<const uint4 *>(wrow + (((4 * half + c4) ^ (n & 7)) << 4));
                    wds[4 * c4 + 0] = p.x;
                    wds[4 * c4 + 1] = p.y;
                    wds[4 * c4 + 2] = p.z;
                    wds[4 * c4 + 3] = p.w;
                }
            }
            // 128 + z_i as a BF16 pair (z_i = clamp(rint(z), 0, 15); a NaN z
            // gives z_i = 0 and reaches the output through the residual)
            uint32_t zpair = SYM ? 0x43084308u : 0x43004300u;  // symmetric INT4: z = 8
            if (zrow) {
                const float zi = fminf(fmaxf(rintf(f16_bits_to_f32(z_tile[n * a.G + g])), 0.0f), 15.0f);
                const uint32_t zb = 0x4300u + static_cast<uint32_t>(zi);
                zpair = zb | (zb << 16);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t cols[32];
                if (wrow_ok) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        // codes 8j..8j+7 of this half (code i at bits 4i..4i+3) ->
                        // BF16 128 + q (the byte q under the byte 0x43) -> q - z_i,
                        // exact; column 4j + i holds codes (8j + 2i, 8j + 2i + 1)
                        const uint32_t w = wds[8 * c + j];
                        const uint32_t lo = w & 0x0F0F0F0Fu;         // q0 q2 q4 q6
                        const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // q1 q3 q5 q7
                        const uint32_t q0123 = __byte_perm(lo, hi, 0x5140);
                        const uint32_t q4567 = __byte_perm(lo, hi, 0x7362);
                        cols[4 * j + 0] = bf16x2_sub(__byte_perm(q0123, 0x43434343u, 0x4140), zpair);
                        cols[4 * j + 1] = bf16x2_sub(__byte_perm(q0123, 0x43434343u, 0x4342), zpair);
                        cols[4 * j + 2] = bf16x2_sub(__byte_perm(q4567, 0x43434343u, 0x4140), zpair);
                        cols[4 * j + 3] = bf16x2_sub(__byte_perm(q4567, 0x43434343u, 0x4342), zpair);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) cols[j] = ONES;  // lanes 28-31: S_g rows
                }
                tmem_st_32x32b_x32(tmem + t_lane + TM_A + ap * 64 + 32 * c, cols);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar.aready[ap]);
                // the box is free once both parities' builders are done with it
                // (with an odd group count the last box is never awaited)
                mbar_arrive(&bar.wempty[ws]);
            }
        }
        // this warp's TMEM stores are complete (waited above, or none issued
        // since the last wait): TMEM may be released as far as it is concerned
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.done);
    } else if (warp >= 4) {
        reg_acquire<kRegEpi>();
        // ------------------------------------------------ group epilogue
        const int q = warp & 3;                // TMEM lane quarter
        const int hc = warp >= 12 ? 1 : 0;     // column half: rows m of X
        const int n = q * RQ + lane;           // output column of this thread (lanes < 28)
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        // this warp's half of the accumulator holds X rows 64 hc .. 64 hc + 63
        // of the tile: none when bm <= 64 and hc = 1 (it only hands the
        // accumulator back)
        const bool has_rows = hc * 64 < bm;
        float y[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) y[j] = 0.0f;
        // warp-uniform waits (one lane per barrier): the shuffles and votes
        // below need the whole warp
        bool ok = mbar_wait_lanes<kHintEpi>(lane == 0 ? &bar.szfull : nullptr, 0, a.status);
        const bool row_ok = lane < RQ && n < rows_n;
        int db = 0, dph = 0;
        for (int g = 0; ok && g < ngroups; ++g) {
            if (!mbar_wait_lanes<kHintEpi>(lane == 0 ? &bar.accfull[db] : nullptr, dph, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float sf = row_ok ? f16_bits_to_f32(s_tile[n * a.G + g]) : 0.0f;
            float zr = 0.0f;  // residual z - z_i (the operand holds q - z_i; 0 when symmetric)
            if (!SYM && row_ok) {
                const float zf = f16_bits_to_f32(z_tile[n * a.G + g]);
                zr = zf - fminf(fmaxf(rintf(zf), 0.0f), 15.0f);
            }
            // warp-uniform: fold S_g in only if some row of this warp needs it
            const bool fold_sg = __any_sync(0xffffffffu, zr != 0.0f);
            const float sc = -sf * zr;
            const uint32_t t_acc = tmem + t_lane + db * 128 + hc * 64;
            // both halves into registers, then release the accumulator at
            // once: the MMAs of group g + DB need it, the arithmetic does not
            if (!has_rows) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.accempty[db]);
                if (++db == DB) {
                    db = 0;
                    dph ^= 1;
                }
                continue;
            }
            uint32_t r[2][32];
            tmem_ld_32x32b_x32(t_acc, r[0]);
            tmem_ld_32x32b_x32(t_acc + 32, r[1]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.accempty[db]);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (fold_sg) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        // lane 28 of every quarter accumulated the row of ones: S_g[m]
                        const float sg = __shfl_sync(0xffffffffu, __uint_as_float(r[c][j]), RQ);
                        y[32 * c + j] = fmaf(sf, __uint_as_float(r[c][j]), fmaf(sc, sg, y[32 * c + j]));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) y[32 * c + j] = fmaf(sf, __uint_as_float(r[c][j]), y[32 * c + j]);
                }
            }
            if (++db == DB) {
                db = 0;
                dph ^= 1;
            }
        }
        if (ok && row_ok) {
            uint16_t *dst = a.Y + static_cast<size_t>(m0 + hc * 64) * a.N + n0 + n;
            const int mrows = min(64, a.M - (m0 + hc * 64));
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (j < mrows) dst[static_cast<size_t>(j) * a.N] = f32_to_bf16_bits(y[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.done);
    }
}


}  // namespace

cudaError_t launch_gemm_int4(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const uint16_t *z,
                             uint16_t *Y, int64_t M, int64_t N, int64_t K, cudaStream_t st, unsigned int *status,
                             const DeviceInfo &dev) {
    if (K > MAX_K) return cudaErrorNotSupported;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    // X rows per tile: M rounded up to 16 below 128, so that the X copies
    // read no rows past M (a zero-filled row costs the copy as much as a
    // loaded one) and the MMAs and the epilogue handle only those rows
    const int bm = M >= BM ? BM : static_cast<int>((M + 15) / 16) * 16;
    const unsigned gx = static_cast<unsigned>((N + BNW - 1) / BNW), gy = static_cast<unsigned>((M + bm - 1) / bm);
    CUtensorMap tmX, tmW;
    {
        // X as BF16 [M, K] seen as [K/64][M][64] (element (k0, row, kb) at byte
        // row * 2K + kb * 128 + 2 k0; K % 128 == 0): box 64 x bm rows x 2, so
        // that one copy brings a group's two 64-K halves (128-byte swizzle).
        // Each TMA copy costs the SM a roughly fixed time, whatever its size.
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(M),
                                    static_cast<cuuint64_t>(K / BK)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, BK * 2};
        const cuuint32_t box[3] = {BK, static_cast<cuuint32_t>(bm), 2};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(X), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // packed codes as bytes [N, K/2]; box of 128 bytes (four K blocks) x 112 rows
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
        const cuuint32_t box[2] = {128, BNW};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(qw), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    GemmArgs a;
    a.s = s;
    a.z = z;
    a.Y = Y;
    a.status = status;
    a.inject = dev.inject;
    a.bm = bm;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.G = static_cast<int>(K / 128);
    a.sz_bytes = (BNW * a.G * 2 + 15) & ~15;  // whole 16-byte chunks of the tile's rows
    // as many X stages (groups of [2][bm rows][128 bytes]) as shared memory
    // allows (3 .. MAX_XP; the MMA issuers step their ring positions by two
    // groups and order their waits by the ring depth)
    const int x_stage = 2 * bm * BK * 2;
    const int tail = WS * W_BYTES + 2 * a.sz_bytes + static_cast<int>(sizeof(Barriers));
    int xp = (dev.max_smem_optin - 1024 - tail) / x_stage;
    if (xp > MAX_XP) xp = MAX_XP;
    if (xp < 3) return cudaErrorNotSupported;
    a.xp = xp;
    a.off_w = OFF_X + xp * x_stage;      // 1024-aligned (x_stage is a multiple of 4 KB)
    a.off_sz = a.off_w + WS * W_BYTES;   // W_BYTES = 14 KB keeps 1024 alignment
    const int smem = 1024 + a.off_sz + 2 * a.sz_bytes + static_cast<int>(sizeof(Barriers));
    // one instance per zero-point mode, each configured once per device
    const int sym = z ? 0 : 1;
    auto kern = sym ? gemm_int4_tc_kernel<true> : gemm_int4_tc_kernel<false>;
    static SmemLimit limit[2];
    auto check_regs = [kern]() -> cudaError_t {
        // the per-role register split (setmaxnreg) must fit in what the block
        // is launched with, or the growing warpgroups would wait for ever
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        const int launch_regs = fa.numRegs;
        if (launch_regs * THREADS < kRegSplit || launch_regs < static_cast<int>(kRegBuild) ||
            launch_regs < static_cast<int>(kRegLight) || launch_regs > static_cast<int>(kRegEpi))
            return cudaErrorNotSupported;
        return cudaSuccess;
    };
    if (cudaError_t e = limit[sym].ensure(reinterpret_cast<const void *>(kern), dev.device, smem, check_regs))
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, gy, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, a);
}

}  // namespace w4
