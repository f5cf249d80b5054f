// A chain of M = 1 INT4 linears in ONE persistent launch ("Lab 5: Gemma4
// end-to-end inference optimisation", sections "CUDA Graph" and "Performance
// analysis": a decode step is hundreds of short bandwidth-bound GEMVs, and
// what separates them -- launch overhead, each grid's ramp and drain -- is
// what costs).
//
//   for each op i in order:  y_i[n] = sum_k x_i[k] * (q_i[n,k] - z_i[n,k/128]) * s_i[n,k/128]
//
// One CTA per SM (a cooperative launch, all resident at once, whenever an op
// of the launch waits for another).  Warp CW, the
// producer, walks every op's rows of this CTA in order and streams their
// packed codes, scales and zeros into the shared-memory stage ring exactly as
// the single GEMV does (gemv_kernel.cuh), without pausing between ops: the
// weights of op i + 1 flow in while op i finishes, because weights never
// depend on an earlier op's output.  When a stage comes back it writes that
// block's outputs; when every stage of op i in this CTA has come back, the
// CTA has finished op i (outputs written, activation read), and the producer
// adds one to done[i] (device-scope release).
//
// The consumers take the ops in the same order.  Before reading op i's
// activation they wait, if op i depends on an earlier op d (it reads what d
// writes, or writes what d reads or writes; found on the host), until done[d]
// equals the grid size, i.e. every CTA has finished op d and so every op
// before it.  Independent ops run back to back with no grid-wide wait.
//
// done[] (count entries) and an exit counter live in caller scratch memory;
// they are zero when a launch starts, and the last CTA to leave resets them
// to zero.
// Every wait is bounded (kWaitLimitNs); a wait that runs out sets the device
// status and its thread leaves, the producer waits for its own copies in
// flight, and the exit counter still resets the scratch.
#include "gemv_kernel.cuh"
#include "kernels.h"

namespace w4 {
namespace {

// 12 consumer warps and the producer: 13 warps, within the 16-warp register
// allocation of 128 registers a thread (17 warps would round up to 20 and
// leave 96, which the op loop around the stage loop does not fit).
constexpr int CW = 16;       // consumer warps
constexpr int RPT = 2;       // most rows per consumer thread per stage

struct ChainMeta {
    long long vrow;  // first row of the block
    int op;
    int rows;
    int soff;        // half-words between the stage's s/z region start and the block's first group
    int pad;
};

struct ChainHeader {
    uint64_t full[kGemvMaxStages];
    uint64_t empty[kGemvMaxStages];
    uint64_t loaded;  // every consumer warp holds the op's activation in registers
    uint64_t sync_b;  // the op's activation converted
    ChainMeta meta[kGemvMaxStages];
    float psum[kGemvMaxStages][2][CW][RPT];  // per-warp row partials, by phase parity
};

// Per-op geometry, computed alike by every role of every CTA.
struct OpGeom {
    int G, half_k, tt_log2, rpt, RB, w_bytes, sz_bytes;
    int64_t begin, end;  // this CTA's rows
};

__device__ __forceinline__ OpGeom op_geom(const ChainOp &o) {
    OpGeom g;
    g.G = o.K >> 7;
    g.half_k = o.K >> 1;
    g.tt_log2 = o.tt_log2;
    g.rpt = o.rpt;
    g.RB = ((CW * 32) >> o.tt_log2) * o.rpt;
    g.w_bytes = g.RB * g.half_k;
    g.sz_bytes = (g.RB * g.G * 2 + 32 + 15) & ~15;
    const unsigned grid = gridDim.x, b = blockIdx.x;
    const unsigned q = static_cast<unsigned>(o.N) / grid, r = static_cast<unsigned>(o.N) % grid;
    g.begin = static_cast<int64_t>(b) * q + (b < r ? b : r);
    g.end = g.begin + q + (b < r ? 1 : 0);
    return g;
}

__device__ __forceinline__ int op_blocks(const ChainOp &o) {
    const OpGeom g = op_geom(o);
    return static_cast<int>((g.end - g.begin + g.RB - 1) / g.RB);
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void red_add_release_gpu(unsigned int *p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int atom_add_acq_rel_gpu(unsigned int *p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *p >= target (a counter other CTAs raise with release
// semantics).  False, with the timeout bit set, when the limit runs out or
// another wait of the device has already timed out.
__device__ bool wait_count(const unsigned int *p, unsigned int target, unsigned int *status) {
    if (ld_acquire_gpu(p) >= target) return true;
    const unsigned long long t0 = global_timer_ns();
#pragma unroll 1
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i) {
            __nanosleep(64);
            if (ld_acquire_gpu(p) >= target) return true;
        }
        if (*reinterpret_cast<volatile unsigned int *>(status) & kDevTimeout) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

template <int NOPS>
struct ChainParams {
    ChainOp ops[NOPS];
    unsigned int *done;    // [count] completion counters, then the exit counter
    unsigned int *status;
    int count;
    int reports;           // some op reports its completion (the counters are used)
    int stages;
    int stage_bytes;       // 128-aligned slot, the largest stage of any op
    int stage_off;         // byte offset of stage 0
    int x_off;             // byte offset of the converted activation
    unsigned int inject;   // test-only injection flags (0 normally)
};

template <int NOPS>
__device__ __forceinline__ void chain_producer(const ChainParams<NOPS> &a, ChainHeader &h, unsigned char *stage0,
                                               int lane) {
    const int S = a.stages;
    const uint64_t pol = policy_evict_first();
    int issued = 0, retired = 0;
    int sig_op = 0;                                   // next op whose completion this CTA reports
    int64_t sig_cum = a.count > 0 ? op_blocks(a.ops[0]) : 0;  // stages of ops 0 .. sig_op
    bool ok = !(a.inject & kInjectStallPipeline);

    auto finalize = [&](int slot, int par, const ChainMeta m) {
        const ChainOp &o = a.ops[m.op];
        const int wpt_log2 = o.tt_log2 - 5;
        const int rpt_log2 = o.rpt - 1;  // rpt 1 or 2
        for (int r = lane; r < m.rows; r += 32) {
            const int team = r >> rpt_log2, rr = r & rpt_log2;
            float acc = 0.0f;
            for (int w = 0; w < (1 << wpt_log2); ++w) acc += h.psum[slot][par][(team << wpt_log2) + w][rr];
            o.y[m.vrow + r] = f32_to_bf16_bits(acc);
        }
    };
    // Report every op whose stages in this CTA have all come back (its
    // outputs are written and its activation was read before its stages
    // were taken), if a later op depends on it; ops are taken in order.  Each
    // lane's release fence orders its own output stores before the count.
    auto report = [&]() {
        while (sig_op < a.count && retired >= sig_cum) {
            if (a.ops[sig_op].report) {
                fence_acq_rel_gpu();
                __syncwarp();
                if (lane == 0) red_add_release_gpu(&a.done[sig_op], 1u);
            }
            if (++sig_op < a.count) sig_cum += op_blocks(a.ops[sig_op]);
        }
    };

    for (int op = 0; ok && op < a.count; ++op) {
        const ChainOp &o = a.ops[op];
        const OpGeom g = op_geom(o);
        const int64_t sz_total = static_cast<int64_t>(o.N) * g.G * 2;  // bytes of the scale (and zero) tensor
        for (int64_t v = g.begin; v < g.end;) {
            const int slot = issued % S;
            const bool recycle = issued >= S;
            const int old_par = ((issued / S) - 1) & 1;
            ChainMeta old{};
            if (recycle) {
                if (!mbar_wait(&h.empty[slot], old_par, a.status)) {
                    ok = false;
                    break;
                }
                old = h.meta[slot];
                __syncwarp();
            }
            const int rows = static_cast<int>(g.end - v < g.RB ? g.end - v : g.RB);
            unsigned char *st = stage0 + slot * a.stage_bytes;
            unsigned char *ss = st + g.w_bytes;
            unsigned char *sz = ss + g.sz_bytes;
            // the block's scale (and zero) rows: one contiguous byte range
            // [b0, b1), copied by its enclosing 16-byte chunks (zero-filled
            // past the tensor's end)
            const uint64_t b0 = static_cast<uint64_t>(v) * g.G * 2;
            const uint64_t b1 = b0 + static_cast<uint64_t>(rows) * g.G * 2;
            const uint64_t lo16 = b0 & ~uint64_t(15);
            if (lane == 0) {
                h.meta[slot].vrow = v;
                h.meta[slot].op = op;
                h.meta[slot].rows = rows;
                h.meta[slot].soff = static_cast<int>((b0 - lo16) >> 1);
                const uint32_t wb = static_cast<uint32_t>(rows) * g.half_k;
                mbar_arrive_expect_tx(&h.full[slot], wb);
                bulk_g2s(st, o.qw + v * g.half_k, wb, &h.full[slot], pol);
            }
            const unsigned char *gs = reinterpret_cast<const unsigned char *>(o.s);
            const unsigned char *gz = reinterpret_cast<const unsigned char *>(o.z);
            for (uint64_t off = lo16 + 16 * static_cast<uint64_t>(lane); off < b1; off += 16 * 32) {
                const uint64_t left = static_cast<uint64_t>(sz_total) - off;
                const uint32_t n = left < 16 ? static_cast<uint32_t>(left) : 16u;
                cp_async_16_zfill(ss + (off - lo16), gs + off, n);
                if (gz) cp_async_16_zfill(sz + (off - lo16), gz + off, n);
            }
            cp_async_arrive_noinc(&h.full[slot]);
            if (recycle) {
                finalize(slot, old_par, old);
                ++retired;
                report();
            }
            v += rows;
            ++issued;
        }
    }
    // the stages still out
    while (ok && retired < issued) {
        const int slot = retired % S, par = (retired / S) & 1;
        if (!mbar_wait(&h.empty[slot], par, a.status)) {
            ok = false;
            break;
        }
        finalize(slot, par, h.meta[slot]);
        ++retired;
        report();
    }
    if (ok) {
        report();  // ops with no rows in this CTA after the last stage
    } else {
        // after a wait ran out: no copy may still be landing when the CTA
        // exits; a stage's full barrier completes on its own copies alone
        for (int it = retired > issued - S ? retired : issued - S; it < issued; ++it)
            mbar_wait(&h.full[it % S], (it / S) & 1, nullptr);
    }
    // the last CTA out returns the counters to zero for the next launch
    // (every CTA has reported everything it will by then)
    if (a.reports) {
        __syncwarp();
        unsigned int prev = 0;
        if (lane == 0) prev = atom_add_acq_rel_gpu(&a.done[a.count], 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == gridDim.x - 1)
            for (int i = lane; i <= a.count; i += 32) a.done[i] = 0u;
    }
}

// The consumers' part of one op: its activation into registers, then its
// nblocks stages, R (= the op's rows per thread) rows each.  Returns false
// when a wait ran out.
template <int R>
__device__ __forceinline__ bool chain_consume_op(const ChainOp &o, int nblocks, ChainHeader &h,
                                              const unsigned char *stage0, const unsigned char *xs, int &slot,
                                              int &phase, int stages, int stage_bytes, unsigned int *status,
                                              int warp, int lane) {
    const int G = o.K >> 7, half_k = o.K >> 1;
    const int w_bytes = (((CW * 32) >> o.tt_log2) * R) * half_k;
    const int team = threadIdx.x >> o.tt_log2;
    const int grp = threadIdx.x & ((1 << o.tt_log2) - 1);  // group of this thread
    const bool valid = grp < G;
    const int gs = valid ? grp : 0;
    const int rot = (grp >> 1) & 3;
    Int4X x;
    int4_load_x(xs, gemv_x_gp(o.K), gs, rot, valid, x);
    __syncwarp();
    if (lane == 0) mbar_arrive(&h.loaded);  // this warp no longer reads the activation region
    const bool sym = o.z == nullptr;
    const int rbase = team * R;
    for (int b = 0; b < nblocks; ++b) {
        if (!mbar_wait(&h.full[slot], phase, status)) return false;
        const unsigned char *st = stage0 + slot * stage_bytes;
        float part[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) part[rr] = 0.0f;
        if (valid) {
            const int soff = h.meta[slot].soff;
            const int sz_bytes = (((CW * 32) >> o.tt_log2) * R * G * 2 + 32 + 15) & ~15;
            const uint16_t *ss = reinterpret_cast<const uint16_t *>(st + w_bytes) + soff;
            const uint16_t *sz = reinterpret_cast<const uint16_t *>(st + w_bytes + sz_bytes) + soff;
            int4_group_rows<R>(x, st, half_k, rbase, gs, rot, ss, sz, sym, G,
                               reinterpret_cast<const uint4 *>(xs) + 16 * gemv_x_gp(o.K) + gs, part);
        }
        const float red = warp_reduce_rows<R>(part, lane);
        if ((lane & (32 / R - 1)) == 0) h.psum[slot][phase][warp][reduced_row<R>(lane)] = red;
        __syncwarp();
        if (lane == 0) mbar_arrive(&h.empty[slot]);
        if (++slot == stages) {
            slot = 0;
            phase ^= 1;
        }
    }
    return true;
}

template <int NOPS>
__global__ void __launch_bounds__((CW + 1) * 32, 1) gemv_chain_kernel(const __grid_constant__ ChainParams<NOPS> a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    ChainHeader &h = *reinterpret_cast<ChainHeader *>(smem);
    unsigned char *stage0 = smem + a.stage_off;
    unsigned char *xs = smem + a.x_off;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&h.full[i], 33);  // producer lane 0 (+ weight bytes) and its 32 cp.async lanes
            mbar_init(&h.empty[i], CW);
        }
        mbar_init(&h.loaded, CW);
        mbar_init(&h.sync_b, CW);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == CW) {
        // the first op's codes into L2 while the previous kernel drains (an L2
        // prefetch cannot hide a later write: L2 is the point of coherence)
        if (lane == 0 && a.count > 0) {
            const OpGeom g = op_geom(a.ops[0]);
            const int64_t rows = g.end - g.begin < 2 * g.RB ? g.end - g.begin : 2 * g.RB;
            const unsigned char *p = a.ops[0].qw + g.begin * g.half_k;
            for (int64_t off = 0; off < rows * g.half_k; off += 32768) {
                const int64_t n = rows * g.half_k - off < 32768 ? rows * g.half_k - off : 32768;
                prefetch_l2_bulk(p + off, static_cast<uint32_t>(n));
            }
        }
        // the scratch counters, activations and outputs follow the stream order
        pdl_wait();
        chain_producer<NOPS>(a, h, stage0, lane);
        return;
    }
    // the first op's first scale and zero rows into L2 while the previous
    // kernel drains (as its codes, above)
    if (a.count > 0) {
        const OpGeom g = op_geom(a.ops[0]);
        const int64_t rows = g.end - g.begin < 2 * g.RB ? g.end - g.begin : 2 * g.RB;
        const uint64_t b0 = static_cast<uint64_t>(g.begin) * g.G * 2, b1 = b0 + static_cast<uint64_t>(rows) * g.G * 2;
        gemv_prefetch_range(a.ops[0].s, b0, b1, threadIdx.x, CW * 32);
        if (a.ops[0].z) gemv_prefetch_range(a.ops[0].z, b0, b1, threadIdx.x, CW * 32);
    }
    pdl_wait();
    if (a.inject & kInjectStallConsumers) return;  // test-only: the producer's waits run out
    int slot = 0, phase = 0, done_ops = 0;  // done_ops: ops this CTA's consumers have taken
    for (int op = 0; op < a.count; ++op) {
        const ChainOp &o = a.ops[op];
        const OpGeom g = op_geom(o);
        if (g.begin >= g.end) continue;  // no rows here (uniform over the CTA)
        // the op this one depends on finished in every CTA (each warp waits
        // for itself; the acquire load and the warp barrier order its reads)
        if (o.dep >= 0) {
            bool met = true;
            if (lane == 0) met = wait_count(&a.done[o.dep], gridDim.x, a.status);
            if (!__shfl_sync(0xffffffffu, met, 0)) return;
        }
        // every warp has copied the previous op's activation into registers
        // (long since, as a rule): the region may be rewritten
        if (done_ops > 0 && !mbar_wait(&h.loaded, (done_ops - 1) & 1, a.status)) return;
        // the activation, converted once per CTA by all consumer warps
        gemv_convert_vector<false, true>(o.x, xs, o.K, warp, CW, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&h.sync_b);
        if (!mbar_wait(&h.sync_b, done_ops & 1, a.status)) return;
        ++done_ops;
        const int nblocks = static_cast<int>((g.end - g.begin + g.RB - 1) / g.RB);
        const bool ok = g.rpt == 2 ? chain_consume_op<2>(o, nblocks, h, stage0, xs, slot, phase, a.stages,
                                                         a.stage_bytes, a.status, warp, lane)
                                   : chain_consume_op<1>(o, nblocks, h, stage0, xs, slot, phase, a.stages,
                                                         a.stage_bytes, a.status, warp, lane);
        if (!ok) return;
    }
}

template <int NOPS>
cudaError_t chain_launch(const ChainOp *ops, int count, unsigned int *done, cudaStream_t st, unsigned int *status,
                         const DeviceInfo &dev) {
    static_assert(sizeof(ChainParams<NOPS>) <= 32000, "kernel parameters");
    ChainParams<NOPS> a{};
    int x_bytes = 0, stage_bytes = 0;
    for (int i = 0; i < count; ++i) {
        a.ops[i] = ops[i];
        const int K = ops[i].K, G = K / 128;
        const int RB = ((CW * 32) >> ops[i].tt_log2) * ops[i].rpt;
        const int sz = (RB * G * 2 + 32 + 15) & ~15;
        const int sb = (RB * (K / 2) + 2 * sz + 127) & ~127;
        stage_bytes = sb > stage_bytes ? sb : stage_bytes;
        x_bytes = gemv_int4_x_bytes(K) > x_bytes ? gemv_int4_x_bytes(K) : x_bytes;
    }
    a.done = done;
    a.status = status;
    a.count = count;
    a.reports = 0;
    for (int i = 0; i < count; ++i) a.reports |= ops[i].report;
    a.inject = dev.inject;
    a.stage_bytes = stage_bytes;
    a.x_off = (static_cast<int>(sizeof(ChainHeader)) + 127) & ~127;
    a.stage_off = (a.x_off + x_bytes + 1023) & ~1023;
    int stages = (dev.max_smem_optin - a.stage_off) / stage_bytes;
    if (stages > kGemvMaxStages) stages = kGemvMaxStages;
    if (stages < 2) return cudaErrorInvalidValue;
    a.stages = stages;
    const int smem = a.stage_off + stages * stage_bytes;
    auto kern = gemv_chain_kernel<NOPS>;
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure(reinterpret_cast<const void *>(kern), dev.device, smem)) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(dev.num_sms));
    cfg.blockDim = dim3((CW + 1) * 32);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // with a dependency inside the launch, CTAs wait on one another's
    // counters, so every CTA must be resident at once: a cooperative launch
    // (it costs the overlap with the previous kernel, so only then)
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.reports ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

void gemv_chain_shape(int64_t K, unsigned char &tt_log2, unsigned char &rpt) {
    // the single GEMV's shape (gemv_dispatch, with its kGemvCW consumer warps):
    // one thread per group, two rows per thread while its stage stays within
    // the stage target -- so that every row is summed in the same order as
    // there, and the results agree bit for bit
    unsigned char l = 5;
    while ((int64_t(1) << l) < K / 128) ++l;
    tt_log2 = l;
    const int64_t teams = (kGemvCW * 32) >> l;
    rpt = (teams * 2 * (K / 2) <= kGemvStageTarget && teams * 2 <= kGemvMaxRB) ? 2 : 1;
}

cudaError_t launch_gemv_chain(const ChainOp *ops, int count, unsigned int *done, cudaStream_t st,
                              unsigned int *status, const DeviceInfo &dev) {
    if (count < 1 || count > kChainMaxOps) return cudaErrorInvalidValue;
    if (count <= 4) return chain_launch<4>(ops, count, done, st, status, dev);
    if (count <= 32) return chain_launch<32>(ops, count, done, st, status, dev);
    return chain_launch<kChainMaxOps>(ops, count, done, st, status, dev);
}

}  // namespace w4
