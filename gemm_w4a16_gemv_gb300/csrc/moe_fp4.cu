// Batched-expert FP4 GEMV for one token:
//   y[i, n] = sum_k x[k] * e2m1(q[ids[i], n, k]) * s[ids[i], n, k/32]
// ("DeepSeek V4 Triton FP4 optimisation in practice": six routed experts per
// token; stacking expert weights on the host cost 20% end to end, so all
// experts are computed in one launch straight from the resident stack).
//
// Same pipeline as the INT4 GEMV: a producer warp streams row blocks of the
// selected experts into a shared-memory ring with cp.async.bulk (scales with
// cp.async), consumer warps keep their K slice of x in registers.  Output rows
// are "virtual rows" v = i * N + n; a row block never crosses an expert
// boundary, so each block is one contiguous range of one expert's matrix.
// The producer reads the expert id of each block from device memory; an id
// outside [0, E) sets the device status and its output rows are written as
// zeros.  E2M1 pairs are decoded with cvt.rn.f16x2.e2m1x2 (exact in FP16).
#include "common.cuh"
#include "kernels.h"

namespace w4 {
namespace {

constexpr int kStages = 4;
constexpr int kStageTarget = 16384;
constexpr int kMaxRB = 32;
constexpr int kHeaderBytes = 4352;

struct MoeArgs {
    const uint16_t *x;
    const uint8_t *qw;
    const uint16_t *s;
    const int32_t *ids;
    uint16_t *y;
    unsigned int *status;
    int64_t E, N;
    int topk, K, G, UPR, RB;
    int w_bytes, s_bytes, stage_bytes;
};

struct BlockMeta {
    int rows;
    int valid;
};

// Two E2M1 codes (one byte; low nibble = even k) -> their values.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2)
        : "r"(byte));
    return __half22float2(*reinterpret_cast<__half2 *>(&h2));
}

__device__ __forceinline__ float2 dot8_fp4(uint32_t w, const float2 *xp, float2 acc) {
    acc = __ffma2_rn(e2m1x2_to_f32x2(w & 0xFFu), xp[0], acc);
    acc = __ffma2_rn(e2m1x2_to_f32x2((w >> 8) & 0xFFu), xp[1], acc);
    acc = __ffma2_rn(e2m1x2_to_f32x2((w >> 16) & 0xFFu), xp[2], acc);
    acc = __ffma2_rn(e2m1x2_to_f32x2(w >> 24), xp[3], acc);
    return acc;
}

// Block sequence of this CTA over virtual rows [begin, end).
struct BlockIter {
    int64_t v, end, N;
    int RB;
    __device__ int next_rows() const {
        const int64_t boundary = (v / N + 1) * N;
        int64_t r = end - v;
        if (boundary - v < r) r = boundary - v;
        if (RB < r) r = RB;
        return static_cast<int>(r);
    }
};

template <int CW, int TT, int UPT>
__global__ void __launch_bounds__((CW + 1) * 32, 2)
moe_fp4_kernel(const MoeArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kStages;
    float *psum = reinterpret_cast<float *>(empty + kStages);  // [kStages][CW][kMaxRB]
    BlockMeta *meta = reinterpret_cast<BlockMeta *>(psum + kStages * CW * kMaxRB);
    unsigned char *stage0 = smem + kHeaderBytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t V = static_cast<int64_t>(a.topk) * a.N;
    const int64_t begin = blockIdx.x * V / gridDim.x;
    const int64_t end = (blockIdx.x + 1) * V / gridDim.x;
    const int half_k = a.K >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 33);
            mbar_init(&empty[i], CW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CW) {
        // ------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        int64_t vrow[kStages];  // first virtual row of the block held in each slot
        constexpr int kWarpsPerTeam = TT / 32;
        const int rpt = a.RB / (CW * 32 / TT);
        auto finalize = [&](int slot) {
            const int rows = meta[slot].rows;
            const bool ok = meta[slot].valid != 0;
            for (int r = lane; r < rows; r += 32) {
                const int w0 = (r / rpt) * kWarpsPerTeam;
                float acc = 0.0f;
                for (int w = w0; w < w0 + kWarpsPerTeam; ++w) acc += psum[(slot * CW + w) * kMaxRB + r];
                a.y[vrow[slot] + r] = ok ? f32_to_bf16_bits(acc) : static_cast<uint16_t>(0);
            }
        };
        BlockIter bi{begin, end, a.N, a.RB};
        int it = 0;
        for (; bi.v < end; ++it) {
            const int slot = it % kStages;
            if (it >= kStages) {
                if (!mbar_wait(&empty[slot], ((it / kStages) - 1) & 1, a.status)) return;
                finalize(slot);
                __syncwarp();
            }
            const int rows = bi.next_rows();
            const int64_t i_slot = bi.v / a.N;
            const int64_t n0 = bi.v - i_slot * a.N;
            const int64_t e = a.ids[i_slot];
            const bool ok = (e >= 0 && e < a.E);
            const int64_t grow = (ok ? e : 0) * a.N + n0;  // row of the [E*N] stack
            unsigned char *st = stage0 + slot * a.stage_bytes;
            uint16_t *ss = reinterpret_cast<uint16_t *>(st + a.w_bytes);
            const uint16_t *gs = a.s + grow * a.G;
            const int ns = rows * a.G;  // even: G is even
            vrow[slot] = bi.v;
            if (lane == 0) {
                if (!ok) atomicOr(a.status, kDevBadExpert);
                meta[slot].rows = rows;
                meta[slot].valid = ok ? 1 : 0;
                const uint32_t wb = ok ? static_cast<uint32_t>(rows) * half_k : 0u;
                mbar_arrive_expect_tx(&full[slot], wb);
                if (ok) bulk_g2s(st, a.qw + grow * half_k, wb, &full[slot], pol);
            }
            if (ok)
                for (int i = lane; i < (ns >> 1); i += 32) cp_async_4(ss + 2 * i, gs + 2 * i);
            cp_async_arrive_noinc(&full[slot]);
            bi.v += rows;
        }
        const int nmine = it;
        const int drain0 = nmine > kStages ? nmine - kStages : 0;
        for (int k = drain0; k < nmine; ++k) {
            if (!mbar_wait(&empty[k % kStages], (k / kStages) & 1, a.status)) return;
            finalize(k % kStages);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    constexpr int TEAMS = CW * 32 / TT;
    const int team = threadIdx.x / TT;
    const int j = threadIdx.x % TT;
    const int RPT = a.RB / TEAMS;

    float2 xr[UPT][16];
    bool valid[UPT];
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
        const int u = j + i * TT;
        valid[i] = u < a.UPR;
        if (valid[i]) {
            const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + 32 * u);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = __ldg(xp + q);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    xr[i][q * 4 + h] = make_float2(bf16_bits_to_f32(w[h] & 0xFFFFu),
                                                   bf16_bits_to_f32(w[h] >> 16));
            }
        } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) xr[i][q] = make_float2(0.0f, 0.0f);
        }
    }

    // Consumers walk the same block sequence as the producer; the number of
    // rows of a block is read from the stage's metadata.
    int64_t v = begin;
    for (int it = 0; v < end; ++it) {
        const int slot = it % kStages;
        if (!mbar_wait(&full[slot], (it / kStages) & 1, a.status)) return;
        const int rows = meta[slot].rows;
        const unsigned char *st = stage0 + slot * a.stage_bytes;
        const uint16_t *ss = reinterpret_cast<const uint16_t *>(st + a.w_bytes);
        if (meta[slot].valid) {
            for (int rr = 0; rr < RPT; ++rr) {
                const int r = team * RPT + rr;
                if (r >= rows) break;
                float part = 0.0f;
#pragma unroll
                for (int i = 0; i < UPT; ++i) {
                    if (!valid[i]) continue;
                    const int u = j + i * TT;
                    const uint4 wv = *reinterpret_cast<const uint4 *>(st + (static_cast<size_t>(r) * a.UPR + u) * 16);
                    const float sf = f16_bits_to_f32(ss[r * a.G + u]);  // one scale per 32 codes
                    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
                    acc0 = dot8_fp4(wv.x, &xr[i][0], acc0);
                    acc1 = dot8_fp4(wv.y, &xr[i][4], acc1);
                    acc0 = dot8_fp4(wv.z, &xr[i][8], acc0);
                    acc1 = dot8_fp4(wv.w, &xr[i][12], acc1);
                    part = fmaf(sf, (acc0.x + acc1.x) + (acc0.y + acc1.y), part);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (lane == 0) psum[(slot * CW + warp) * kMaxRB + r] = part;
            }
        }
        v += rows;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
}

template <int TT, int UPT>
cudaError_t launch_one(const MoeArgs &a, int smem, cudaStream_t st, const DeviceInfo &dev) {
    constexpr int CW = 8;
    auto kern = moe_fp4_kernel<CW, TT, UPT>;
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
    const int64_t V = static_cast<int64_t>(a.topk) * a.N;
    int64_t ctas = static_cast<int64_t>(dev.num_sms) * occupancy[d];
    if (ctas > V) ctas = V;
    if (ctas < 1) ctas = 1;
    kern<<<static_cast<unsigned>(ctas), (CW + 1) * 32, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_moe_fp4(const uint16_t *x, const uint8_t *qw,
                           const uint16_t *s, const int32_t *ids, int topk,
                           uint16_t *y, int64_t E, int64_t N, int64_t K,
                           cudaStream_t st, unsigned int *status,
                           const DeviceInfo &dev) {
    constexpr int CW = 8;
    const int UPR = static_cast<int>(K / 32);
    struct Cfg {
        int TT, UPT;
    };
    const Cfg cands[] = {{32, 2}, {64, 2}, {128, 2}, {256, 2},
                         {32, 1}, {64, 1}, {128, 1}, {256, 1}};
    Cfg best = {0, 0};
    int best_cover = 1 << 30;
    for (const Cfg &c : cands) {
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
    MoeArgs a;
    a.x = x;
    a.qw = qw;
    a.s = s;
    a.ids = ids;
    a.y = y;
    a.status = status;
    a.E = E;
    a.N = N;
    a.topk = topk;
    a.K = static_cast<int>(K);
    a.G = static_cast<int>(K / 32);
    a.UPR = UPR;
    a.RB = teams * rpt;
    if (a.RB > kMaxRB) return cudaErrorInvalidValue;
    a.w_bytes = a.RB * row_bytes;
    a.s_bytes = ((a.RB * a.G * 2) + 15) & ~15;
    a.stage_bytes = (a.w_bytes + a.s_bytes + 127) & ~127;
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
