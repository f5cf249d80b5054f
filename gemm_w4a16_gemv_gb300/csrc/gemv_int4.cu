// M = 1 decode GEMV with INT4 asymmetric group-128 weights:
//   y[n] = sum_k x[k] * (q[n,k] - z[n,k/128]) * s[n,k/128]
// ("Lab 5: Gemma4 end-to-end inference optimisation", section "INT4 fused
// GEMV": the packed weight is read once, unpacked in registers, scaled and
// zero-shifted per group and dotted with the activation, never written back).
//
// Design (HBM-bound; every packed byte is read exactly once):
//  * one producer warp per CTA streams contiguous row blocks of the packed
//    matrix into a ring of shared-memory stages with cp.async.bulk (the
//    matrix is row-major, so RB full rows are one contiguous range), and the
//    matching scale / zero rows with 4-byte cp.async; both complete on the
//    stage's "full" mbarrier;
//  * consumer warps own fixed 32-code K slices ("units") of every row, so
//    their slice of the activation stays in registers for the whole launch;
//  * a 32-bit word of 8 codes is unpacked with shifts and AND/OR into
//    binary32 numbers 128 + q/2 (even k) and 128 + 8q (odd k); the activation
//    is stored pre-scaled by 2 and 1/8, so each packed FMA adds q*x plus a
//    constant bias term; the bias sum and the zero-point term z * sum(x) are
//    removed once per unit, and the group scale is applied once per unit;
//  * per-row partials are reduced with warp shuffles and shared-memory
//    atomics; the producer writes the finished BF16 outputs of a stage when
//    it recycles the stage.
// Every mbarrier wait is bounded; on timeout the device status is set and the
// CTA returns.
#include "common.cuh"
#include "kernels.h"

namespace w4 {
namespace {

constexpr int kStages = 4;
constexpr int kStageTarget = 16384;  // packed weight bytes per stage
constexpr int kMaxRB = 32;           // rows per stage, upper bound
constexpr int kHeaderBytes = 4352;   // barriers + per-warp row partials

struct GemvArgs {
    const uint16_t *x;
    const uint8_t *qw;
    const uint16_t *s;
    const uint16_t *z;
    uint16_t *y;
    unsigned int *status;
    int64_t N;
    int K, G, UPR, RB;
    int w_bytes;      // packed-weight region of a stage (RB * K/2)
    int sz_bytes;     // one of the s / z regions of a stage (16-aligned)
    int stage_bytes;  // whole stage (128-aligned)
};

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// Eight codes of one word against eight pre-scaled activations (see above).
__device__ __forceinline__ float2 dot8(uint32_t w, const float2 *xp, float2 acc) {
    const uint32_t t0 = w << 15, t1 = w << 7, t2 = w >> 1, t3 = w >> 9;
    acc = __ffma2_rn(make_float2(as_f((t0 & 0x00078000u) | 0x43000000u),
                                 as_f((t0 & 0x00780000u) | 0x43000000u)),
                     xp[0], acc);
    acc = __ffma2_rn(make_float2(as_f((t1 & 0x00078000u) | 0x43000000u),
                                 as_f((t1 & 0x00780000u) | 0x43000000u)),
                     xp[1], acc);
    acc = __ffma2_rn(make_float2(as_f((t2 & 0x00078000u) | 0x43000000u),
                                 as_f((t2 & 0x00780000u) | 0x43000000u)),
                     xp[2], acc);
    acc = __ffma2_rn(make_float2(as_f((t3 & 0x00078000u) | 0x43000000u),
                                 as_f((t3 & 0x00780000u) | 0x43000000u)),
                     xp[3], acc);
    return acc;
}

__device__ __forceinline__ int64_t even_floor(int64_t v) { return v & ~int64_t(1); }

// Rows [begin, end) of this CTA: an even-aligned share of N.
__device__ __forceinline__ void cta_rows(int64_t N, int64_t &begin, int64_t &end) {
    const int64_t C = gridDim.x, c = blockIdx.x;
    begin = even_floor(c * N / C);
    end = (c == C - 1) ? N : even_floor((c + 1) * N / C);
}

template <int CW, int TT, int UPT>
__global__ void __launch_bounds__((CW + 1) * 32, 2)
gemv_int4_kernel(const GemvArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kStages;
    float *psum = reinterpret_cast<float *>(empty + kStages);  // [kStages][CW][kMaxRB]
    unsigned char *stage0 = smem + kHeaderBytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int64_t row_begin, row_end;
    cta_rows(a.N, row_begin, row_end);
    const int nmine = static_cast<int>((row_end - row_begin + a.RB - 1) / a.RB);
    const int half_k = a.K >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 33);  // producer lane 0 (+tx) and 32 cp.async lanes
            mbar_init(&empty[i], CW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CW) {
        // ------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        constexpr int kWarpsPerTeam = TT / 32;
        const int rpt = a.RB / (CW * 32 / TT);
        auto finalize = [&](int it) {
            const int slot = it % kStages;
            const int64_t row0 = row_begin + static_cast<int64_t>(it) * a.RB;
            const int rows = static_cast<int>(row_end - row0 < a.RB ? row_end - row0 : a.RB);
            for (int r = lane; r < rows; r += 32) {
                // warps of the team that owns row r, summed in a fixed order
                const int w0 = (r / rpt) * kWarpsPerTeam;
                float acc = 0.0f;
                for (int w = w0; w < w0 + kWarpsPerTeam; ++w) acc += psum[(slot * CW + w) * kMaxRB + r];
                a.y[row0 + r] = f32_to_bf16_bits(acc);
            }
        };
        for (int it = 0; it < nmine; ++it) {
            const int slot = it % kStages;
            if (it >= kStages) {
                if (!mbar_wait(&empty[slot], ((it / kStages) - 1) & 1, a.status)) return;
                finalize(it - kStages);
                __syncwarp();
            }
            const int64_t row0 = row_begin + static_cast<int64_t>(it) * a.RB;
            const int rows = static_cast<int>(row_end - row0 < a.RB ? row_end - row0 : a.RB);
            unsigned char *st = stage0 + slot * a.stage_bytes;
            uint16_t *ss = reinterpret_cast<uint16_t *>(st + a.w_bytes);
            uint16_t *sz = reinterpret_cast<uint16_t *>(st + a.w_bytes + a.sz_bytes);
            const uint16_t *gs = a.s + row0 * a.G;
            const uint16_t *gz = a.z + row0 * a.G;
            const int nsz = rows * a.G;
            if (lane == 0) {
                if (nsz & 1) {  // odd tail: one half-word copied synchronously
                    ss[nsz - 1] = gs[nsz - 1];
                    sz[nsz - 1] = gz[nsz - 1];
                }
                const uint32_t wb = static_cast<uint32_t>(rows) * half_k;
                mbar_arrive_expect_tx(&full[slot], wb);
                bulk_g2s(st, a.qw + row0 * half_k, wb, &full[slot], pol);
            }
            for (int i = lane; i < (nsz >> 1); i += 32) {
                cp_async_4(ss + 2 * i, gs + 2 * i);
                cp_async_4(sz + 2 * i, gz + 2 * i);
            }
            cp_async_arrive_noinc(&full[slot]);
        }
        const int drain0 = nmine > kStages ? nmine - kStages : 0;
        for (int it = drain0; it < nmine; ++it) {
            if (!mbar_wait(&empty[it % kStages], (it / kStages) & 1, a.status)) return;
            finalize(it);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    constexpr int TEAMS = CW * 32 / TT;
    const int team = threadIdx.x / TT;
    const int j = threadIdx.x % TT;
    const int RPT = a.RB / TEAMS;

    float2 xr[UPT][16];
    float cu[UPT], xu[UPT];
    bool valid[UPT];
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
        const int u = j + i * TT;
        valid[i] = u < a.UPR;
        float c = 0.0f, sx = 0.0f;
        if (valid[i]) {
            const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + 32 * u);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = __ldg(xp + q);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float xe = bf16_bits_to_f32(w[h] & 0xFFFFu);  // even k
                    const float xo = bf16_bits_to_f32(w[h] >> 16);      // odd k
                    xr[i][q * 4 + h] = make_float2(xe * 2.0f, xo * 0.125f);
                    c += 256.0f * xe + 16.0f * xo;
                    sx += xe + xo;
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) xr[i][q] = make_float2(0.0f, 0.0f);
        }
        cu[i] = c;
        xu[i] = sx;
    }

    for (int it = 0; it < nmine; ++it) {
        const int slot = it % kStages;
        if (!mbar_wait(&full[slot], (it / kStages) & 1, a.status)) return;
        const int64_t row0 = row_begin + static_cast<int64_t>(it) * a.RB;
        const int rows = static_cast<int>(row_end - row0 < a.RB ? row_end - row0 : a.RB);
        const unsigned char *st = stage0 + slot * a.stage_bytes;
        const uint16_t *ss = reinterpret_cast<const uint16_t *>(st + a.w_bytes);
        const uint16_t *sz = reinterpret_cast<const uint16_t *>(st + a.w_bytes + a.sz_bytes);
        for (int rr = 0; rr < RPT; ++rr) {
            const int r = team * RPT + rr;
            if (r >= rows) break;  // uniform across the warp (TT >= 32)
            float part = 0.0f;
#pragma unroll
            for (int i = 0; i < UPT; ++i) {
                if (!valid[i]) continue;
                const int u = j + i * TT;
                const uint4 wv = *reinterpret_cast<const uint4 *>(st + (static_cast<size_t>(r) * a.UPR + u) * 16);
                const int g = u >> 2;
                const float sf = f16_bits_to_f32(ss[r * a.G + g]);
                const float zf = f16_bits_to_f32(sz[r * a.G + g]);
                float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
                acc0 = dot8(wv.x, &xr[i][0], acc0);
                acc1 = dot8(wv.y, &xr[i][4], acc1);
                acc0 = dot8(wv.z, &xr[i][8], acc0);
                acc1 = dot8(wv.w, &xr[i][12], acc1);
                float t = ((acc0.x + acc1.x) + (acc0.y + acc1.y)) - cu[i];
                t = fmaf(-zf, xu[i], t);
                part = fmaf(sf, t, part);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) psum[(slot * CW + warp) * kMaxRB + r] = part;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
}

struct Config {
    int TT, UPT;
};

template <int TT, int UPT>
cudaError_t launch_one(const GemvArgs &a, int smem, cudaStream_t st, const DeviceInfo &dev) {
    constexpr int CW = 8;
    auto kern = gemv_int4_kernel<CW, TT, UPT>;
    static int configured_smem[64] = {0};
    static int occupancy[64] = {0};
    const int d = dev.device & 63;
    if (configured_smem[d] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured_smem[d] = smem;
        occupancy[d] = 0;
    }
    if (occupancy[d] == 0) {
        int occ = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, (CW + 1) * 32, smem);
        if (e != cudaSuccess) return e;
        occupancy[d] = occ > 0 ? occ : 1;
    }
    int64_t ctas = static_cast<int64_t>(dev.num_sms) * occupancy[d];
    const int64_t max_ctas = (a.N + 1) / 2;  // at least two rows each
    if (ctas > max_ctas) ctas = max_ctas;
    if (ctas < 1) ctas = 1;
    kern<<<static_cast<unsigned>(ctas), (CW + 1) * 32, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_int4(const uint16_t *x, const uint8_t *qw,
                             const uint16_t *s, const uint16_t *z, uint16_t *y,
                             int64_t N, int64_t K, cudaStream_t st,
                             unsigned int *status, const DeviceInfo &dev) {
    constexpr int CW = 8;
    const int UPR = static_cast<int>(K / 32);
    // threads per row (TT) and units per thread (UPT): cover UPR with the
    // least idle slots, preferring two units per thread (half the reductions).
    const Config cands[] = {{32, 2}, {64, 2}, {128, 2}, {256, 2},
                            {32, 1}, {64, 1}, {128, 1}, {256, 1}};
    Config best = {0, 0};
    int best_cover = 1 << 30;
    for (const Config &c : cands) {
        const int cover = c.TT * c.UPT;
        if (cover >= UPR && cover < best_cover) {
            best = c;
            best_cover = cover;
        }
    }
    if (best.TT == 0) return cudaErrorInvalidValue;
    const int teams = CW * 32 / best.TT;
    const int row_bytes = static_cast<int>(K / 2);
    int rpt = kStageTarget / (teams * row_bytes);
    if (rpt < 1) rpt = 1;
    if (rpt > 4) rpt = 4;
    if ((teams * rpt) & 1) rpt = (rpt == 1) ? 2 : rpt - 1;
    GemvArgs a;
    a.x = x;
    a.qw = qw;
    a.s = s;
    a.z = z;
    a.y = y;
    a.status = status;
    a.N = N;
    a.K = static_cast<int>(K);
    a.G = static_cast<int>(K / 128);
    a.UPR = UPR;
    a.RB = teams * rpt;
    if (a.RB > kMaxRB) return cudaErrorInvalidValue;
    a.w_bytes = a.RB * row_bytes;
    a.sz_bytes = ((a.RB * a.G * 2) + 15) & ~15;
    a.stage_bytes = (a.w_bytes + 2 * a.sz_bytes + 127) & ~127;
    const int smem = kHeaderBytes + kStages * a.stage_bytes;
    switch (best.TT * 10 + best.UPT) {
        case 322: return launch_one<32, 2>(a, smem, st, dev);
        case 642: return launch_one<64, 2>(a, smem, st, dev);
        case 1282: return launch_one<128, 2>(a, smem, st, dev);
        case 2562: return launch_one<256, 2>(a, smem, st, dev);
        case 321: return launch_one<32, 1>(a, smem, st, dev);
        case 641: return launch_one<64, 1>(a, smem, st, dev);
        case 1281: return launch_one<128, 1>(a, smem, st, dev);
        case 2561: return launch_one<256, 1>(a, smem, st, dev);
    }
    return cudaErrorInvalidValue;
}

}  // namespace w4
