// The M = 1 streaming GEMV pipeline shared by the INT4 decode GEMV and the
// FP4 batched-expert GEMV.
//
//   INT4: y[v]       = sum_k x[k] * (q[v,k] - z[v,k/128]) * s[v,k/128]
//   FP4 : y[i*N + n] = sum_k x[k] * e2m1(q[ids[i],n,k]) * s[ids[i],n,k/32]
//
// One persistent CTA per SM.  Warp CW is the producer: it walks this CTA's
// output rows ("virtual rows" v; for FP4 v = i*N + n) in blocks of at most RB
// rows that never cross an expert boundary, and for each block issues one
// cp.async.bulk of the block's packed rows (one contiguous range of the
// row-major matrix) plus 4-byte cp.async copies of the block's scale (and
// zero) rows, all completing on the stage's "full" mbarrier.  A ring of
// `stages` shared-memory stages keeps up to ~150 KB of weights in flight.
//
// Warps 0..CW-1 consume.  The activation vector is converted once per CTA,
// cooperatively, into f16x2 pairs with an exact power-of-two scale per
// 32-element unit (gemv_common.cuh) and parked in shared memory; each thread
// then keeps the pairs of its own units in registers.  Threads form teams of
// TT threads; a team owns RPT rows of every stage and each of its threads
// owns UPT 32-code units of those rows.  Per-row partials are reduced across
// the warp with a transposed butterfly and across the team's warps by the
// producer, in a fixed order (so results are bitwise reproducible), when it
// recycles the stage; it then writes the BF16 outputs.  All waits are bounded.
#pragma once

#include "common.cuh"
#include "gemv_common.cuh"

namespace w4 {

constexpr int kGemvMaxStages = 8;
constexpr int kGemvMaxRB = 32;

struct GemvParams {
    const uint16_t *x;
    const uint8_t *qw;
    const uint16_t *s;
    const uint16_t *z;      // INT4 only
    const int32_t *ids;     // FP4 only
    uint16_t *y;
    unsigned int *status;
    int64_t rows_per_slot;  // FP4: N (one expert's rows); INT4: N
    int64_t V;              // virtual rows in total (INT4: N; FP4: topk * N)
    int64_t E;              // FP4: number of experts
    int K, G, UPR, RB, stages;
    int w_bytes;            // packed weights of a stage (RB * K/2)
    int sz_bytes;           // one scale (or zero) region of a stage, 16-aligned
    int stage_bytes;        // 128-aligned
    int x_off;              // byte offset of the staged activations
    int stage_off;          // byte offset of stage 0
};

struct StageMeta {
    long long vrow;  // first virtual row of the block
    int rows;
    int valid;       // FP4: expert id in range
};

template <int CW, int RPT>
struct GemvHeader {
    uint64_t full[kGemvMaxStages];
    uint64_t empty[kGemvMaxStages];
    StageMeta meta[kGemvMaxStages];
    float psum[kGemvMaxStages][2][CW][RPT];  // per-warp row partials, by phase parity
};

// Per-unit constants: INT4 bias sum, effective activation sum; scale undo.
struct UnitConst {
    float c, xs, pw, pad;
};

__device__ __forceinline__ int64_t gemv_even_floor(int64_t v) { return v & ~int64_t(1); }

// Rows of the block starting at virtual row v (this CTA's range ends at end).
__device__ __forceinline__ int gemv_block_rows(int64_t v, int64_t end, int64_t per_slot, int RB) {
    const int64_t boundary = (v / per_slot + 1) * per_slot;
    int64_t r = end - v;
    if (boundary - v < r) r = boundary - v;
    if (RB < r) r = RB;
    return static_cast<int>(r);
}

template <bool FP4, int CW, int TT, int UPT, int RPT>
__device__ __forceinline__ void gemv_producer(const GemvParams &a, GemvHeader<CW, RPT> &h,
                                              unsigned char *stage0, int64_t begin, int64_t end,
                                              int lane) {
    constexpr int WPT = TT / 32;  // warps per team
    const int half_k = a.K >> 1;
    const uint64_t pol = policy_evict_first();
    // Write the outputs of a finished block.  Its metadata is copied out before
    // the slot is reused, and its partials sit in the half of psum indexed by
    // the block's phase parity, which the slot's next block does not touch.
    auto finalize = [&](int slot, int par, const StageMeta m) {
        for (int r = lane; r < m.rows; r += 32) {
            const int team = r / RPT, rr = r - team * RPT;
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < WPT; ++w) acc += h.psum[slot][par][team * WPT + w][rr];
            a.y[m.vrow + r] = m.valid ? f32_to_bf16_bits(acc) : static_cast<uint16_t>(0);
        }
    };
    int slot = 0, phase = 0, issued = 0;
    for (int64_t v = begin; v < end; ++issued) {
        const bool recycle = issued >= a.stages;
        StageMeta old{};
        if (recycle) {
            if (!mbar_wait(&h.empty[slot], phase ^ 1, a.status)) return;
            old = h.meta[slot];
            __syncwarp();
        }
        const int rows = gemv_block_rows(v, end, a.rows_per_slot, a.RB);
        int64_t src_row = v;
        bool ok = true;
        if (FP4) {
            const int64_t i_slot = v / a.rows_per_slot;
            const int64_t e = a.ids[i_slot];
            ok = (e >= 0 && e < a.E);
            src_row = (ok ? e : 0) * a.rows_per_slot + (v - i_slot * a.rows_per_slot);
        }
        unsigned char *st = stage0 + slot * a.stage_bytes;
        uint16_t *ss = reinterpret_cast<uint16_t *>(st + a.w_bytes);
        uint16_t *sz = reinterpret_cast<uint16_t *>(st + a.w_bytes + a.sz_bytes);
        const uint16_t *gs = a.s + src_row * a.G;
        const uint16_t *gz = FP4 ? nullptr : a.z + src_row * a.G;
        const int nsz = rows * a.G;
        if (lane == 0) {
            if (!ok) atomicOr(a.status, kDevBadExpert);
            h.meta[slot].vrow = v;
            h.meta[slot].rows = rows;
            h.meta[slot].valid = ok ? 1 : 0;
            if (!FP4 && (nsz & 1)) {  // odd tail: one half-word copied synchronously
                ss[nsz - 1] = gs[nsz - 1];
                sz[nsz - 1] = gz[nsz - 1];
            }
            const uint32_t wb = ok ? static_cast<uint32_t>(rows) * half_k : 0u;
            mbar_arrive_expect_tx(&h.full[slot], wb);
            if (ok) bulk_g2s(st, a.qw + src_row * half_k, wb, &h.full[slot], pol);
        }
        if (ok) {
            for (int i = lane; i < (nsz >> 1); i += 32) {
                cp_async_4(ss + 2 * i, gs + 2 * i);
                if (!FP4) cp_async_4(sz + 2 * i, gz + 2 * i);
            }
        }
        cp_async_arrive_noinc(&h.full[slot]);
        // the next copy is in flight; now finish the block this slot held
        if (recycle) finalize(slot, phase ^ 1, old);
        v += rows;
        if (++slot == a.stages) {
            slot = 0;
            phase ^= 1;
        }
    }
    // drain: finish the last min(stages, issued) blocks
    const int first = issued > a.stages ? issued - a.stages : 0;
    for (int it = first; it < issued; ++it) {
        const int sl = it % a.stages;
        if (!mbar_wait(&h.empty[sl], (it / a.stages) & 1, a.status)) return;
        finalize(sl, (it / a.stages) & 1, h.meta[sl]);
    }
}

// Cooperative activation staging: one thread per 32-element unit writes the
// unit's 16 f16x2 pairs and its constants to shared memory.
template <bool FP4>
__device__ __forceinline__ void gemv_stage_x(const GemvParams &a, uint32_t *xh_s, UnitConst *xc_s, int tid,
                                             int nthreads) {
    for (int u = tid; u < a.UPR; u += nthreads) {
        uint32_t xb[16];
        load_x_unit(a.x + 32 * u, xb);
        const int e = unit_exponent(xb);
        const float inv = pow2f(14 - e);
        UnitConst uc;
        uc.pw = pow2f(e - 14);
        uc.pad = 0.0f;
        float c = 0.0f, xs = 0.0f;
        uint32_t out[16];
        if (FP4) {
            // natural pairs (x[2i], x[2i+1]), matching the E2M1 byte decode
#pragma unroll
            for (int q = 0; q < 16; ++q)
                out[q] = pack_half2(bf16_elem(xb, 2 * q) * inv, bf16_elem(xb, 2 * q + 1) * inv);
        } else {
            // INT4 unpack order for word m: (8m, 8m+4), (8m+1, 8m+5)/16,
            // (8m+2, 8m+6), (8m+3, 8m+7)/16 -- the /16 pairs meet codes that
            // the unpack leaves multiplied by 16
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float f = (q & 1) ? 0.0625f : 1.0f;
                    const float v0 = bf16_elem(xb, 8 * m + q) * inv * f;
                    const float v1 = bf16_elem(xb, 8 * m + q + 4) * inv * f;
                    out[4 * m + q] = pack_half2(v0, v1);
                    c += v0 + v1;                                   // times the 1024 bias below
                    xs += (q & 1) ? 16.0f * (v0 + v1) : (v0 + v1);  // activation each product sees
                }
            }
        }
        uc.c = 1024.0f * c;
        uc.xs = xs;
        uint4 *dst = reinterpret_cast<uint4 *>(xh_s + 16 * u);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
        xc_s[u] = uc;
    }
}

template <bool FP4, int CW, int TT, int UPT, int RPT>
__global__ void __launch_bounds__((CW + 1) * 32, 1) gemv_stream_kernel(const GemvParams a) {
    using Header = GemvHeader<CW, RPT>;
    extern __shared__ __align__(1024) unsigned char smem[];
    Header &h = *reinterpret_cast<Header *>(smem);
    uint32_t *xh_s = reinterpret_cast<uint32_t *>(smem + a.x_off);                // [UPR][16]
    UnitConst *xc_s = reinterpret_cast<UnitConst *>(smem + a.x_off + a.UPR * 64);  // [UPR]
    unsigned char *stage0 = smem + a.stage_off;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // This CTA's virtual rows.  INT4 ranges start on even rows, so every block
    // start is even and the 4-byte copies of scale/zero rows stay aligned when
    // K/128 is odd.
    int64_t begin = blockIdx.x * a.V / gridDim.x;
    int64_t end = (blockIdx.x + 1) * a.V / gridDim.x;
    if (!FP4) {
        begin = gemv_even_floor(begin);
        end = (blockIdx.x + 1 == gridDim.x) ? a.V : gemv_even_floor(end);
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&h.full[i], 33);  // producer lane 0 (+tx) and 32 cp.async lanes
            mbar_init(&h.empty[i], CW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CW) {
        gemv_producer<FP4, CW, TT, UPT, RPT>(a, h, stage0, begin, end, lane);
        return;
    }

    gemv_stage_x<FP4>(a, xh_s, xc_s, threadIdx.x, CW * 32);
    named_bar_sync(1, CW * 32);

    const int team = threadIdx.x / TT;
    const int j = threadIdx.x % TT;
    uint32_t xh[UPT][16];
    float cu[UPT], xu[UPT], pw[UPT];
    bool valid[UPT];
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
        const int u = j + i * TT;
        valid[i] = u < a.UPR;
        const int us = valid[i] ? u : 0;
        const uint4 *src = reinterpret_cast<const uint4 *>(xh_s + 16 * us);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 t = src[q];
            xh[i][4 * q] = t.x;
            xh[i][4 * q + 1] = t.y;
            xh[i][4 * q + 2] = t.z;
            xh[i][4 * q + 3] = t.w;
        }
        const UnitConst uc = xc_s[us];
        cu[i] = uc.c;
        xu[i] = uc.xs;
        pw[i] = valid[i] ? uc.pw : 0.0f;
    }

    const int rbase = team * RPT;
    int slot = 0, phase = 0;
    for (int64_t v = begin; v < end;) {
        if (!mbar_wait(&h.full[slot], phase, a.status)) return;
        const int rows = h.meta[slot].rows;
        const unsigned char *st = stage0 + slot * a.stage_bytes;
        const uint16_t *ss = reinterpret_cast<const uint16_t *>(st + a.w_bytes);
        const uint16_t *sz = reinterpret_cast<const uint16_t *>(st + a.w_bytes + a.sz_bytes);
        float part[RPT];
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr) part[rr] = 0.0f;
#pragma unroll
        for (int i = 0; i < UPT; ++i) {
            if (!valid[i]) continue;
            const int u = j + i * TT;
            uint4 wv[RPT];
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr)
                wv[rr] = *reinterpret_cast<const uint4 *>(st + (static_cast<size_t>(rbase + rr) * a.UPR + u) * 16);
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr) {
                float lo = 0.0f, hi = 0.0f;
                const uint32_t words[4] = {wv[rr].x, wv[rr].y, wv[rr].z, wv[rr].w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t w = words[m];
                    if (FP4) {
                        mfma_f16x2(e2m1x2_to_f16x2(w), xh[i][4 * m + 0], lo, hi);
                        mfma_f16x2(e2m1x2_to_f16x2(w >> 8), xh[i][4 * m + 1], lo, hi);
                        mfma_f16x2(e2m1x2_to_f16x2(w >> 16), xh[i][4 * m + 2], lo, hi);
                        mfma_f16x2(e2m1x2_to_f16x2(w >> 24), xh[i][4 * m + 3], lo, hi);
                    } else {
                        // two codes per logic op: binary16 1024 + q and 1024 + 16q
                        const uint32_t w8 = w >> 8;
                        mfma_f16x2((w & 0x000F000Fu) | 0x64006400u, xh[i][4 * m + 0], lo, hi);
                        mfma_f16x2((w & 0x00F000F0u) | 0x64006400u, xh[i][4 * m + 1], lo, hi);
                        mfma_f16x2((w8 & 0x000F000Fu) | 0x64006400u, xh[i][4 * m + 2], lo, hi);
                        mfma_f16x2((w8 & 0x00F000F0u) | 0x64006400u, xh[i][4 * m + 3], lo, hi);
                    }
                }
                if (FP4) {
                    const float sf = f16_bits_to_f32(ss[(rbase + rr) * a.G + u]) * pw[i];  // one scale per unit
                    part[rr] = fmaf(sf, lo + hi, part[rr]);
                } else {
                    const int g = (rbase + rr) * a.G + (u >> 2);
                    const float sf = f16_bits_to_f32(ss[g]) * pw[i];
                    const float zf = f16_bits_to_f32(sz[g]);
                    float t = (lo + hi) - cu[i];
                    t = fmaf(-zf, xu[i], t);
                    part[rr] = fmaf(sf, t, part[rr]);
                }
            }
        }
        const float red = warp_reduce_rows<RPT>(part, lane);
        if ((lane & (32 / RPT - 1)) == 0) h.psum[slot][phase][warp][reduced_row<RPT>(lane)] = red;
        __syncwarp();
        if (lane == 0) mbar_arrive(&h.empty[slot]);
        v += rows;
        if (++slot == a.stages) {
            slot = 0;
            phase ^= 1;
        }
    }
}

// Host side: pick the team shape for K, size the stages, launch one CTA per SM.
struct GemvShape {
    int TT, UPT, RPT;
};

inline GemvShape gemv_choose_shape(int CW, int UPR, int row_bytes, int stage_target) {
    // Threads per row (TT) and units per thread (UPT): cover a row's UPR
    // units with the fewest idle slots, preferring two units per thread.
    const GemvShape cands[] = {{32, 2, 0}, {64, 2, 0}, {128, 2, 0}, {256, 2, 0}, {32, 1, 0}};
    GemvShape best = {0, 0, 0};
    int best_cover = 1 << 30;
    for (const GemvShape &c : cands) {
        if (c.TT > CW * 32) continue;
        const int cover = c.TT * c.UPT;
        if (cover >= UPR && cover < best_cover) {
            best = c;
            best_cover = cover;
        }
    }
    if (best.TT == 0) return best;
    const int teams = CW * 32 / best.TT;
    best.RPT = (teams * 4 * row_bytes <= stage_target) ? 4 : 2;
    if (teams * best.RPT > kGemvMaxRB) best.RPT = 2;
    return best;
}

constexpr int kGemvCW = 16;             // consumer warps per CTA
constexpr int kGemvStageTarget = 32768; // packed weight bytes per stage (upper aim)

template <bool FP4, int TT, int UPT, int RPT>
cudaError_t gemv_launch(GemvParams a, cudaStream_t st, int device, int num_sms, int max_smem) {
    constexpr int CW = kGemvCW;
    auto kern = gemv_stream_kernel<FP4, CW, TT, UPT, RPT>;
    const int header = (static_cast<int>(sizeof(GemvHeader<CW, RPT>)) + 127) & ~127;
    a.x_off = header;
    const int x_bytes = a.UPR * 64 + a.UPR * static_cast<int>(sizeof(UnitConst));
    a.stage_off = (a.x_off + x_bytes + 1023) & ~1023;
    int stages = (max_smem - a.stage_off) / a.stage_bytes;
    if (stages > kGemvMaxStages) stages = kGemvMaxStages;
    if (stages < 2) return cudaErrorInvalidValue;
    a.stages = stages;
    const int smem = a.stage_off + stages * a.stage_bytes;
    static int configured[64] = {0};
    const int d = device & 63;
    if (configured[d] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[d] = smem;
    }
    int64_t ctas = num_sms;
    const int64_t max_ctas = (a.V + 1) / 2;  // at least two rows each
    if (ctas > max_ctas) ctas = max_ctas;
    if (ctas < 1) ctas = 1;
    kern<<<static_cast<unsigned>(ctas), (CW + 1) * 32, smem, st>>>(a);
    return cudaGetLastError();
}

// Fill the stage geometry of `a` for K and launch the matching instance.
template <bool FP4>
cudaError_t gemv_dispatch(GemvParams a, cudaStream_t st, int device, int num_sms, int max_smem) {
    a.UPR = a.K / 32;
    const int row_bytes = a.K / 2;
    const GemvShape sh = gemv_choose_shape(kGemvCW, a.UPR, row_bytes, kGemvStageTarget);
    if (sh.TT == 0) return cudaErrorInvalidValue;
    a.RB = (kGemvCW * 32 / sh.TT) * sh.RPT;  // even: RPT is 2 or 4
    if (a.RB > kGemvMaxRB) return cudaErrorInvalidValue;
    a.w_bytes = a.RB * row_bytes;
    a.sz_bytes = ((a.RB * a.G * 2) + 15) & ~15;
    a.stage_bytes = (a.w_bytes + (FP4 ? 1 : 2) * a.sz_bytes + 127) & ~127;
#define W4_GEMV_CASE(TT_, UPT_)                                                                   \
    if (sh.TT == TT_ && sh.UPT == UPT_)                                                           \
        return sh.RPT == 4 ? gemv_launch<FP4, TT_, UPT_, 4>(a, st, device, num_sms, max_smem)     \
                           : gemv_launch<FP4, TT_, UPT_, 2>(a, st, device, num_sms, max_smem);
    W4_GEMV_CASE(32, 2)
    W4_GEMV_CASE(64, 2)
    W4_GEMV_CASE(128, 2)
    W4_GEMV_CASE(256, 2)
    W4_GEMV_CASE(32, 1)
#undef W4_GEMV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace w4
