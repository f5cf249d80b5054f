// Batched-expert FP4 GEMM for M tokens, each routed to topk experts
// ("DeepSeek V4 Triton FP4 optimisation in practice": the fused FP4
// dequantise-and-multiply expert GEMMs; M > 1 is the prefill / batched case):
//
//   Y[m, j, n] = sum_k X[m, k] * e2m1(q[e, n, k]) * s[e, n, k/32],  e = ids[m, j]
//
// Three launches on the caller's stream, all state in caller scratch memory:
//  1. route (one CTA): counts the (token, slot) pairs of each expert, gives
//     every valid pair a position in its expert's contiguous row list, and
//     writes the tile table (an expert's rows in tiles of up to 128); an id
//     outside [0, E) sets the device status;
//  2. gather: copies each routed token row into the scratch as binary16,
//     scaled by a power of two per token so that its largest |x| lands in
//     [2^14, 2^15) (exact for every value within 2^29 of that maximum); the
//     output rows of invalid ids are written as zeros;
//  3. the GEMM on the tcgen05 tensor cores: one persistent CTA per SM,
//     looping over the work items (tile, 128 weight rows), so that the
//     weight stream runs on from one item into the next with no CTA launch,
//     setup, pipeline fill or drain between them (each cost about a fifth of
//     an item's time when every item was a CTA of its own).  Builder warps
//     decode the E2M1 codes exactly to binary16
//     (cvt.rn.f16x2.e2m1x2) and multiply by the group scale in binary16 --
//     the weight e2m1 * s rounded once to binary16, a relative error of at
//     most 2^-11 (the only rounding of the operands) -- into the A operand in
//     tensor memory; the gathered token rows are the B operand (TMA, 128-byte
//     swizzle).  The tile has few token rows (the MMA's N is 16 for a
//     typical expert), and MMAs issued by one thread run one after another at
//     about 100-150 SM cycles each whatever N is, while MMAs from different
//     warps into different accumulators overlap.  So issuer warps -- 4
//     while the largest tile has at most 32 rows, 2 up to 64, else 1 -- take
//     turns by 128-K chunk, each into an FP32 accumulator of its own; four epilogue warps sum them, undo each
//     token's power-of-two scale, round to BF16 and scatter the rows to
//     their (token, slot) places while the next item's MMAs run into the
//     other accumulator set.
// Every wait is bounded; on a timeout the status word is set, each role
// still performs the arrivals the others wait for, and tensor memory is
// released only after the MMAs issued have completed.
#include "common.cuh"
#include "gemv_common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace w4 {
namespace {

constexpr int BR = 128;               // weight rows per CTA (the MMA's M; TMEM lanes)
constexpr int BT = 128;               // token rows per tile at most (the MMA's N)
constexpr int CK = 128;               // K per chunk: one A stage, one X stage
constexpr int SCK = 256;              // K per weight stage: 128 code bytes and 8 scales per row
constexpr int XS_MAX = 8;             // X stages: a multiple of the issuer count, so that each
                                      // issuer waits on stages of its own chunks only (in order)
constexpr int WS_MAX = 12;            // weight stages (codes + scales), as many as fit
constexpr int BG = 2;                 // builder groups: chunk c is built by group c mod 2
constexpr int AP = 4;                 // TMEM operand stages (64 columns each), two per group
constexpr int MAX_ISS = 4;            // MMA issuer warps (each with its own accumulator)
constexpr int NXMAPS = BT / 16;        // token tensor maps, one per tile height 16, 32, ..., 128
constexpr int W_STAGE = BR * 128;     // 16 KB of packed codes
constexpr int S_STAGE = BR * 16;      // 2 KB of scales
// Shared memory holds the X ring (stages of 256 bytes per token row of the
// largest tile: 8 stages for tiles of up to 32 rows, 4 beyond) and as many
// weight stages as fit after it: the weight ring keeps the HBM reads in
// flight.
constexpr int POOL = 208 * 1024;
constexpr int THREADS = 640;          // 20 warps: 0 weights TMA, 1 tokens TMA, 2-5 MMA, 6 TMEM,
                                      // 8-15 builders, 16-19 epilogue
constexpr int ISS0 = 2;               // first issuer warp
constexpr int BW0 = 8;                // first builder warp (warp & 3 = its TMEM lane quarter)
constexpr int EW0 = 16;               // first epilogue warp (warp & 3 = its TMEM lane quarter)
constexpr int NEW = 4;                // epilogue warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_ACC = 0;        // two accumulator sets of n_iss x (largest tile's N) <= 128 columns
constexpr uint32_t TM_A = 256;        // operand stages after them
constexpr int ROUTE_THREADS = 1024;
constexpr int GATHER_THREADS = 256;

struct MoeTile {
    int expert;
    int row0;   // first row of the tile in the gathered list
    int rows;   // 1 .. BT
    int pad;
};

// Scratch layout (byte offsets, 256-aligned), a function of P = M * topk,
// E and K only.
struct MoeScratch {
    int64_t tiles_off, perm_off, posof_off, scale_off, xg_off, total;
    int tmax;
};

__host__ __device__ inline int64_t align256(int64_t v) { return (v + 255) & ~int64_t(255); }

__host__ __device__ inline MoeScratch moe_scratch_layout(int64_t P, int64_t E, int64_t K) {
    MoeScratch l;
    l.tmax = static_cast<int>((P + BT - 1) / BT + (E < P ? E : P));
    l.tiles_off = 256;  // the tile count and the largest tile's rows live at offsets 0 and 4
    l.perm_off = align256(l.tiles_off + 16 * static_cast<int64_t>(l.tmax));
    l.posof_off = align256(l.perm_off + 4 * P);
    l.scale_off = align256(l.posof_off + 4 * P);
    l.xg_off = align256(l.scale_off + 4 * P);
    l.total = align256(l.xg_off + 2 * P * K);
    return l;
}

// ------------------------------------------------------------ 1. routing
// Exclusive prefix sum of one value per thread over the routing CTA; `total`
// receives the sum of all of them.  ws: ROUTE_THREADS / 32 ints of shared
// memory (free again when it returns).
__device__ __forceinline__ int route_exclusive_sum(int v, int *ws, int &total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;  // inclusive within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = ws[lane];  // ROUTE_THREADS / 32 == 32 warp sums
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, d);
            if (lane >= d) t += y;
        }
        ws[lane] = t;  // inclusive over the warps
    }
    __syncthreads();
    const int before = w > 0 ? ws[w - 1] : 0;
    total = ws[ROUTE_THREADS / 32 - 1];
    __syncthreads();
    return before + x - v;
}

// One CTA.  cnt[e]: pairs of expert e; off[e]: first position of its rows.
__global__ void __launch_bounds__(ROUTE_THREADS) moe_route_kernel(const int32_t *__restrict__ ids, int P, int E,
                                                                  unsigned char *scratch, unsigned int *status) {
    extern __shared__ int sm[];
    int *cnt = sm;           // [E]
    int *off = sm + E;       // [E]
    int *cur = sm + 2 * E;   // [E]
    const MoeScratch l = moe_scratch_layout(P, E, 0);
    MoeTile *tiles = reinterpret_cast<MoeTile *>(scratch + l.tiles_off);
    int *perm = reinterpret_cast<int *>(scratch + l.perm_off);
    int *posof = reinterpret_cast<int *>(scratch + l.posof_off);
    pdl_wait();
    pdl_launch_dependents();  // the gather's CTAs may start; they wait for this grid before reading
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = cur[e] = 0;
    __syncthreads();
    bool bad = false;
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int e = ids[p];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else bad = true;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, kDevBadExpert);
    // The tile table, experts in order: block-wide exclusive prefix sums of
    // the experts' row counts (off[e]) and tile counts (its first tile), one
    // expert per thread in chunks of the CTA's width, each thread writing its
    // expert's tiles (rows in tiles of BT); the tile count and the largest
    // tile's rows go to the scratch header.
    __shared__ int ws[ROUTE_THREADS / 32];
    __shared__ int max_rows;
    if (threadIdx.x == 0) max_rows = 0;
    int row_carry = 0, tile_carry = 0, my_max = 0;
    for (int e0 = 0; e0 < E; e0 += ROUTE_THREADS) {  // uniform over the CTA
        const int e = e0 + static_cast<int>(threadIdx.x);
        const int c = e < E ? cnt[e] : 0;
        const int ntl = (c + BT - 1) / BT;
        int rows_total, tiles_total;
        const int roff = row_carry + route_exclusive_sum(c, ws, rows_total);
        const int toff = tile_carry + route_exclusive_sum(ntl, ws, tiles_total);
        if (e < E) {
            off[e] = roff;
            for (int j = 0; j < ntl; ++j) {
                MoeTile tl;
                tl.expert = e;
                tl.row0 = roff + j * BT;
                tl.rows = c - j * BT < BT ? c - j * BT : BT;
                tl.pad = 0;
                tiles[toff + j] = tl;
            }
            my_max = max(my_max, c < BT ? c : BT);
        }
        row_carry += rows_total;
        tile_carry += tiles_total;
    }
    atomicMax(&max_rows, my_max);
    __syncthreads();
    if (threadIdx.x == 0) {
        reinterpret_cast<int *>(scratch)[0] = tile_carry;
        reinterpret_cast<int *>(scratch)[1] = max_rows;
    }
    // positions: within an expert in arrival order (each output row is
    // computed on its own, so the order does not change any result)
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int e = ids[p];
        int pos = -1;
        if (e >= 0 && e < E) {
            pos = off[e] + atomicAdd(&cur[e], 1);
            perm[pos] = p;
        }
        posof[p] = pos;
    }
}

// --------------------------------------------------------- 2. gathering
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    return m;
}
// 8 BF16 values times inv (a power of two), each rounded to binary16, in order
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 v, float inv) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(bf16_bits_to_f32(w[i] & 0xFFFFu) * inv, bf16_bits_to_f32(w[i] >> 16) * inv);
        o[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// One CTA per (token, slot) pair p = m * topk + j: the token's row, times
// 2^(14 - e) for its largest |x| in [2^e, 2^(e+1)), into binary16 at the
// pair's position.  NB > 0: the row is read once, each thread holding its NB
// blocks of 8 values (K <= 8 NB GATHER_THREADS); NB = 0: any K, read twice.
template <int NB>
__global__ void __launch_bounds__(GATHER_THREADS) moe_gather_kernel(const uint16_t *__restrict__ X, int topk, int P,
                                                                    int E, int K, int64_t N, uint16_t *Y,
                                                                    unsigned char *scratch) {
    const MoeScratch l = moe_scratch_layout(P, E, K);
    const int p = blockIdx.x;
    pdl_launch_dependents();  // the GEMM's CTAs may start; they wait for this grid before reading
    pdl_wait();               // the routing (and X) follow the stream order
    // K % 256 == 0: rows of whole 16-byte blocks, 16-byte aligned.  The
    // token's row is requested before the pair's position (which only says
    // where the row goes), so that the two loads' latencies overlap.
    const uint4 *x = reinterpret_cast<const uint4 *>(X + static_cast<int64_t>(p / topk) * K);
    const int nb = K / 8;
    uint4 xv[NB > 0 ? NB : 1];
    if constexpr (NB > 0) {
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int b = threadIdx.x + j * GATHER_THREADS;
            xv[j] = b < nb ? x[b] : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    const int pos = reinterpret_cast<const int *>(scratch + l.posof_off)[p];  // uniform over the CTA
    if (pos < 0) {
        // an expert id out of range: its output row is zeros
        for (int64_t n = threadIdx.x; n < N; n += blockDim.x) Y[p * N + n] = 0;
        return;
    }
    uint4 *xg = reinterpret_cast<uint4 *>(scratch + l.xg_off) + static_cast<int64_t>(pos) * (K / 8);
    // largest |x| of the token (BF16 magnitude bit patterns order as values)
    __shared__ uint32_t red[GATHER_THREADS / 32];
    uint32_t m = 0;
    if constexpr (NB > 0) {
#pragma unroll
        for (int j = 0; j < NB; ++j) m = max(m, bf16x8_absmax_bits(xv[j]));
    } else {
        for (int b = threadIdx.x; b < nb; b += GATHER_THREADS) m = max(m, bf16x8_absmax_bits(x[b]));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0;
#pragma unroll
    for (int w = 0; w < GATHER_THREADS / 32; ++w) m = max(m, red[w]);
    const int e = exponent_of_absmax(m);  // 2^e <= max|x| < 2^(e+1)
    const float inv = pow2f(14 - e);      // max|x| * inv in [2^14, 2^15): binary16 holds it
    if constexpr (NB > 0) {
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int b = threadIdx.x + j * GATHER_THREADS;
            if (b >= nb) break;
            xg[b] = bf16x8_to_f16x8(xv[j], inv);
        }
    } else {
        for (int b = threadIdx.x; b < nb; b += GATHER_THREADS) xg[b] = bf16x8_to_f16x8(x[b], inv);
    }
    if (threadIdx.x == 0) reinterpret_cast<float *>(scratch + l.scale_off)[pos] = pow2f(e - 14);
}

// --------------------------------------------------------------- 3. GEMM
struct MoeGemmArgs {
    const unsigned char *scratch;
    uint16_t *Y;
    unsigned int *status;
    int P, E, N, K, nchunks;
    unsigned int inject;
};

// One 3-D view of the gathered token rows per tile height h = 16 (i + 1):
// [K/64][P][64] binary16, box 64 x h x 2, so that one TMA copy brings a
// chunk's h rows x 128 K (both 64-K halves of the 128-byte swizzle).  Every
// TMA copy costs the SM a fixed time whatever its size (measured at about
// 0.14 us each on GB300 with the weight stream running), so the ring moves
// each chunk with as few copies as its shape allows.
struct MoeXMaps {
    CUtensorMap m[NXMAPS];
};

struct MoeBarriers {
    uint64_t xfull[XS_MAX], xempty[XS_MAX];
    uint64_t wfull[WS_MAX], wempty[WS_MAX];
    uint64_t aready[AP], aempty[AP];
    uint64_t accfull[2];   // an item's accumulators complete (n_iss arrivals), by item parity
    uint64_t accempty[2];  // ... read by the epilogue warps (NEW arrivals)
    uint64_t drained;      // every MMA issued has completed (n_iss arrivals, at the end)
    uint64_t done;         // the epilogue warps finished (NEW arrivals)
    uint32_t tmem_holder;
};

// Eight E2M1 codes (the four bytes of w) times a binary16 scale pair -> four
// binary16 pairs, o[i] from byte i, low half from its low nibble (even k):
// decode exact, one rounding.  The word is split into its bytes by one
// vector move, so no shift or mask precedes a conversion.
__device__ __forceinline__ void e2m1x8_times(uint32_t w, uint32_t s2, uint32_t *o) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 h0, b0;\n\tcvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 h2, b2;\n\tcvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
        "mul.rn.f16x2 %0, h0, %5;\n\tmul.rn.f16x2 %1, h1, %5;\n\t"
        "mul.rn.f16x2 %2, h2, %5;\n\tmul.rn.f16x2 %3, h3, %5;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w), "r"(s2));
}

// One persistent CTA per SM loops over the work items (tile t, block b of 128
// weight rows), b fastest.  Every ring runs on across the items (its slot
// and phase from a counter over all of this CTA's chunks or stages); the
// accumulators alternate by item parity, so the epilogue warps drain item s
// while the MMAs of item s + 1 run.  The layout (X stage rows, accumulator
// columns, the issuer count, the ring depths) is set per launch from the
// largest tile; each item loads only its own tile's token rows and
// multiplies with its own N.
__global__ void __launch_bounds__(THREADS, 1)
moe_fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ MoeXMaps xm, const MoeGemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    MoeBarriers &bar = *reinterpret_cast<MoeBarriers *>(smem + POOL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the routing: read after the routing launch has finished (stream order)
    pdl_wait();
    const MoeScratch l = moe_scratch_layout(a.P, a.E, a.K);
    const int ntiles = reinterpret_cast<const int *>(a.scratch)[0];
    const int maxrows = reinterpret_cast<const int *>(a.scratch)[1];
    const MoeTile *tiles = reinterpret_cast<const MoeTile *>(a.scratch + l.tiles_off);
    const int nblk = (a.N + BR - 1) / BR;
    const int total = ntiles * nblk;
    if (static_cast<int>(blockIdx.x) >= total) return;  // uniform over the CTA
    const int nitems = (total - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                       static_cast<int>(gridDim.x);
    // the largest tile sets the layout (X stage rows, accumulator columns);
    // each item loads its own tile's rows and multiplies with its own N
    const int nmax = ((maxrows + 15) / 16) * 16;
    const int nch = a.nchunks;  // even (K % 256 == 0)
    // issuers: as many as two accumulator sets fit in 256 columns; they take
    // turns by chunk within an item, so their count divides the chunks
    int n_iss = nmax <= 32 ? MAX_ISS : (nmax <= 64 ? 2 : 1);
    if (nch % n_iss != 0) n_iss = 2;
    const int x_stage = 2 * nmax * 128;
    const int xs_n = nmax <= 32 ? 8 : 4;  // a multiple of n_iss
    const int off_w = xs_n * x_stage;
    int ws_n = (POOL - off_w) / (W_STAGE + S_STAGE);
    ws_n = ws_n < WS_MAX ? ws_n : WS_MAX;
    const int off_s = off_w + ws_n * W_STAGE;
    const int nsc = a.K / SCK;  // weight stages per item

    if (threadIdx.x == 0) {
        for (int i = 0; i < xs_n; ++i) {
            mbar_init(&bar.xfull[i], 1);
            mbar_init(&bar.xempty[i], 1);
        }
        for (int i = 0; i < ws_n; ++i) {
            mbar_init(&bar.wfull[i], 1);
            mbar_init(&bar.wempty[i], 8);  // the stage's two chunks, four builder warps each
        }
        for (int i = 0; i < AP; ++i) {
            mbar_init(&bar.aready[i], 4);  // the 4 builder warps of the chunk's group
            mbar_init(&bar.aempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.accfull[i], n_iss);
            mbar_init(&bar.accempty[i], NEW);
        }
        mbar_init(&bar.drained, n_iss);
        mbar_init(&bar.done, NEW);
        fence_barrier_init();
    }
    if (warp == 6) {  // this warp allocates tensor memory and frees it at the end
        tmem_alloc(&bar.tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_holder;

    if (warp == 0) {
        // ---------------------------------------- codes and scales (TMA)
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            tma_prefetch_desc(&tmW);
            tma_prefetch_desc(&tmS);
            const int nissue = (a.inject & kInjectStallPipeline) ? 0 : nitems;
            int issued = 0;
            bool ok = true;
            for (int it = 0; ok && it < nissue; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
                const MoeTile tile = tiles[item / nblk];
                // rows past the stack's end read as zeros; rows of the next
                // expert (blocks ending past N) are computed and not stored
                const int wrow0 = tile.expert * a.N + (item % nblk) * BR;
                for (int sc = 0; sc < nsc; ++sc, ++issued) {
                    const int ws = issued % ws_n;
                    if (issued >= ws_n && !mbar_wait(&bar.wempty[ws], ((issued / ws_n) - 1) & 1, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar.wfull[ws], W_STAGE + S_STAGE);
                    tma_load_2d_hint(smem + off_w + ws * W_STAGE, &tmW, sc * 128, wrow0, &bar.wfull[ws], pol);
                    tma_load_2d_hint(smem + off_s + ws * S_STAGE, &tmS, sc * 8, wrow0, &bar.wfull[ws], pol);
                }
            }
            // no copy in flight when the CTA exits
            for (int i = issued > ws_n ? issued - ws_n : 0; i < issued; ++i)
                mbar_wait(&bar.wfull[i % ws_n], (i / ws_n) & 1, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------ token rows (TMA)
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            for (int i = 0; i < NXMAPS; ++i) tma_prefetch_desc(&xm.m[i]);
            const int nissue = (a.inject & kInjectStallPipeline) ? 0 : nitems;
            int issued = 0;
            bool ok = true;
            for (int it = 0; ok && it < nissue; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
                const MoeTile tile = tiles[item / nblk];
                const int nt = ((tile.rows + 15) / 16) * 16;  // rows loaded: the item's MMA N
                const CUtensorMap *map = &xm.m[nt / 16 - 1];
                for (int c = 0; c < nch; ++c, ++issued) {
                    const int xs = issued % xs_n;
                    if (issued >= xs_n && !mbar_wait(&bar.xempty[xs], ((issued / xs_n) - 1) & 1, a.status)) {
                        ok = false;
                        break;
                    }
                    // the stage holds [2][nt][128 bytes]: the two 64-K halves of the chunk
                    mbar_arrive_expect_tx(&bar.xfull[xs], 2 * nt * 128);
                    tma_load_3d_hint(smem + xs * x_stage, map, 0, tile.row0, 2 * c, &bar.xfull[xs], pol);
                }
            }
            for (int i = issued > xs_n ? issued - xs_n : 0; i < issued; ++i)
                mbar_wait(&bar.xfull[i % xs_n], (i / xs_n) & 1, nullptr);
        }
    } else if (warp >= ISS0 && warp < ISS0 + n_iss) {
        // ------------------------------------------------ MMA issuers
        // issuer j takes the chunks c = j mod n_iss of each item into
        // accumulator j of the item's set
        const int j = warp - ISS0;
        bool ok = !(a.inject & kInjectStallConsumers);
        for (int it = 0; ok && it < nitems; ++it) {
            const int set = it & 1;
            const int item = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
            const int nt = ((tiles[item / nblk].rows + 15) / 16) * 16;  // this item's MMA N
            const uint32_t idesc = idesc_kind_f16(BR, nt, 0u);            // FP16 x FP16 -> FP32, M = 128
            // the epilogue has read this set's accumulators of item it - 2
            if (it >= 2 && !mbar_wait_lanes(lane == 0 ? &bar.accempty[set] : nullptr, ((it >> 1) - 1) & 1,
                                            a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_acc = tmem + TM_ACC + static_cast<uint32_t>(set * 128 + j * nmax);
            for (int c = j; c < nch; c += n_iss) {
                const int gc = it * nch + c;
                const int ap = gc % AP, xs = gc % xs_n;
                uint64_t *wbar = nullptr;
                uint32_t par = 0;
                if (lane == 0) {
                    wbar = &bar.aready[ap];
                    par = (gc / AP) & 1;
                } else if (lane == 1) {
                    wbar = &bar.xfull[xs];
                    par = (gc / xs_n) & 1;
                }
                if (!mbar_wait_lanes(wbar, par, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t b_addr = smem_u32(smem + xs * x_stage);
#pragma unroll
                for (int k = 0; k < CK / 16; ++k)
                    umma_f16_tmem_a_w(d_acc, tmem + TM_A + ap * 64 + 8 * k,
                                      smem_desc_sw128_kmajor(b_addr + (k >> 2) * (nt * 128) + 32 * (k & 3)), idesc,
                                      (c != j) || (k != 0));
                umma_commit_w(&bar.xempty[xs]);
                umma_commit_w(&bar.aempty[ap]);
                __syncwarp();
            }
            // the item's accumulators are complete once its MMAs have
            // completed (after a timeout too, so that the epilogue's wait ends)
            umma_commit_w(&bar.accfull[set]);
            __syncwarp();
        }
        umma_commit_w(&bar.drained);
        __syncwarp();
    } else if (warp == 6) {
        // tensor memory is freed only after every MMA has completed and the
        // epilogue has read the accumulators
        mbar_wait(&bar.drained, 0, nullptr);
        mbar_wait(&bar.done, 0, a.status);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    } else if (warp >= BW0 && warp < EW0) {
        // -------------------------------------------- operand builders
        const int q = warp & 3;            // TMEM lane quarter: weight rows 32 q .. 32 q + 31
        const int grp = (warp - BW0) >> 2;  // chunks grp, grp + 2, ... of every item
        const int r = q * 32 + lane;       // weight row of this thread
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        bool ok = true;
        for (int it = 0; ok && it < nitems; ++it) {
            for (int c = grp; c < nch; c += BG) {
                const int gc = it * nch + c;
                const int gs = gc >> 1, ws = gs % ws_n, half = c & 1, ap = gc % AP;
                uint64_t *wbar = nullptr;
                uint32_t wpar = 0;
                if (lane == 0) {
                    wbar = &bar.wfull[ws];
                    wpar = (gs / ws_n) & 1;
                } else if (lane == 1 && gc >= AP) {
                    wbar = &bar.aempty[ap];
                    wpar = ((gc - AP) / AP) & 1;
                }
                if (!mbar_wait_lanes(wbar, wpar, a.status)) {
                    ok = false;
                    break;
                }
                // this row's 64 code bytes of the chunk (16-byte chunks 4 half
                // + 0..3 of the swizzled row, chunk j at j ^ (r mod 8)) and its
                // four group scales (8 per 256-K stage)
                const unsigned char *wrow = smem + off_w + ws * W_STAGE + r * 128;
                uint32_t wds[16];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(wrow + (((4 * half + c4) ^ (r & 7)) << 4));
                    wds[4 * c4] = v.x;
                    wds[4 * c4 + 1] = v.y;
                    wds[4 * c4 + 2] = v.z;
                    wds[4 * c4 + 3] = v.w;
                }
                const uint4 sv = *reinterpret_cast<const uint4 *>(smem + off_s + ws * S_STAGE + r * 16);
                const uint32_t s01 = half ? sv.z : sv.x, s23 = half ? sv.w : sv.y;  // groups 4 half + 0..3
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    // 64 codes (groups 2 cc, 2 cc + 1 of the chunk) -> 32 columns
                    uint32_t cols[32];
#pragma unroll
                    for (int g2 = 0; g2 < 2; ++g2) {
                        const uint32_t sg =
                            cc ? (g2 ? s23 >> 16 : s23 & 0xFFFFu) : (g2 ? s01 >> 16 : s01 & 0xFFFFu);
                        const uint32_t s2 = sg | (sg << 16);
#pragma unroll
                        for (int i = 0; i < 4; ++i) e2m1x8_times(wds[8 * cc + 4 * g2 + i], s2, &cols[16 * g2 + 4 * i]);
                    }
                    tmem_st_32x32b_x32(tmem + t_lane + TM_A + ap * 64 + 32 * cc, cols);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar.aready[ap]);
                    mbar_arrive(&bar.wempty[ws]);
                }
            }
        }
    } else if (warp >= EW0) {
        // ----------------------------------------------------- epilogue
        // the sum of the item's n_iss accumulators per 16-column piece, each
        // token's power-of-two scale undone, scattered to (token, slot) rows
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        const float *rowscale = reinterpret_cast<const float *>(a.scratch + l.scale_off);
        const int *perm = reinterpret_cast<const int *>(a.scratch + l.perm_off);
        for (int it = 0; it < nitems; ++it) {
            const int item = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
            const MoeTile tile = tiles[item / nblk];
            const int n0 = (item % nblk) * BR;
            const int set = it & 1;
            if (!mbar_wait_lanes(lane == 0 ? &bar.accfull[set] : nullptr, (it >> 1) & 1, a.status)) break;
            tc_fence_after();
            const bool nok = n0 + r < a.N;
            for (int p = 0; 16 * p < tile.rows; ++p) {
                float acc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
                for (int jj = 0; jj < n_iss; ++jj) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(tmem + t_lane + TM_ACC + static_cast<uint32_t>(set * 128 + jj * nmax + 16 * p),
                                       v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(v[i]);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int col = 16 * p + i;  // token row of the tile
                    if (col < tile.rows && nok) {
                        const int pos = tile.row0 + col;
                        a.Y[static_cast<int64_t>(perm[pos]) * a.N + n0 + r] = f32_to_bf16_bits(acc[i] * rowscale[pos]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.accempty[set]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.done);
    }
}

}  // namespace

int64_t moe_fp4_gemm_scratch(int64_t P, int64_t E, int64_t K) { return moe_scratch_layout(P, E, K).total; }

cudaError_t launch_moe_fp4_gemm(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const int32_t *ids, int M,
                                int topk, uint16_t *Y, int64_t E, int64_t N, int64_t K, void *scratch,
                                cudaStream_t st, unsigned int *status, const DeviceInfo &dev) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int P = M * topk;
    const MoeScratch l = moe_scratch_layout(P, E, K);
    unsigned char *scr = static_cast<unsigned char *>(scratch);
    // 1. routing
    {
        const int smem = static_cast<int>(3 * E * sizeof(int));
        static SmemLimit limit;
        if (cudaError_t e = limit.ensure(reinterpret_cast<const void *>(moe_route_kernel), dev.device, smem)) return e;
    }
    // the three launches go with programmatic stream serialisation: each may
    // start while the previous launch of the stream finishes and waits for it
    // (griddepcontrol.wait) before touching global memory
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(ROUTE_THREADS);
        cfg.dynamicSmemBytes = static_cast<size_t>(3 * E * sizeof(int));
        cfg.stream = st;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        if (cudaError_t e = cudaLaunchKernelEx(&cfg, moe_route_kernel, ids, P, static_cast<int>(E), scr, status))
            return e;
    }
    // 2. gathering
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(P));
        cfg.blockDim = dim3(GATHER_THREADS);
        cfg.stream = st;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        const int per_thread = static_cast<int>((K / 8 + GATHER_THREADS - 1) / GATHER_THREADS);
        auto gk = per_thread <= 2 ? moe_gather_kernel<2>
                  : per_thread <= 4 ? moe_gather_kernel<4>
                  : per_thread <= 8 ? moe_gather_kernel<8>
                                    : moe_gather_kernel<0>;
        if (cudaError_t e = cudaLaunchKernelEx(&cfg, gk, X, topk, P, static_cast<int>(E), static_cast<int>(K), N, Y, scr))
            return e;
    }
    // 3. the GEMM
    CUtensorMap tmW, tmS;
    MoeXMaps xm;
    {
        // packed codes as bytes [E*N, K/2]: box 128 bytes (256 codes) x 128 rows, 128-byte swizzle
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(E * N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
        const cuuint32_t box[2] = {128, BR};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(qw), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // scales as binary16 [E*N, K/32]: box 8 (16 bytes, one 256-K stage) x 128 rows
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 32), static_cast<cuuint64_t>(E * N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 32) * 2};
        const cuuint32_t box[2] = {8, BR};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tmS, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(s), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // gathered token rows, binary16 [P, K] seen as [K/64][P][64] (element
        // (k0, row, kb) at byte row * 2K + kb * 128 + 2 k0): box 64 x h x 2,
        // 128-byte swizzle, h = 16, 32, ..., 128
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(P), static_cast<cuuint64_t>(K / 64)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
        const cuuint32_t estr[3] = {1, 1, 1};
        for (int i = 0; i < NXMAPS; ++i) {
            const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(16 * (i + 1)), 2};
            if (enc(&xm.m[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, scr + l.xg_off, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
    }
    MoeGemmArgs a;
    a.scratch = scr;
    a.Y = Y;
    a.status = status;
    a.P = P;
    a.E = static_cast<int>(E);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.nchunks = static_cast<int>(K / CK);
    a.inject = dev.inject;
    const int smem = 1024 + POOL + static_cast<int>(sizeof(MoeBarriers));
    if (smem > dev.max_smem_optin) return cudaErrorNotSupported;
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure(reinterpret_cast<const void *>(moe_fp4_gemm_kernel), dev.device, smem)) return e;
    // one persistent CTA per SM (at most one per possible work item)
    const int64_t items_max = static_cast<int64_t>(l.tmax) * ((N + BR - 1) / BR);
    const unsigned grid = static_cast<unsigned>(items_max < dev.num_sms ? items_max : dev.num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_fp4_gemm_kernel, tmW, tmS, xm, a);
}

}  // namespace w4
