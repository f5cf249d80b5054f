// The M = 1 streaming GEMV pipeline shared by the INT4 decode GEMV and the
// FP4 batched-expert GEMV.
//
//   INT4: y[v]       = sum_k x[k] * (q[v,k] - z[v,k/128]) * s[v,k/128]
//   FP4 : y[i*N + n] = sum_k x[k] * e2m1(q[ids[i],n,k]) * s[ids[i],n,k/32]
//
// One persistent CTA per SM, launched with programmatic stream serialisation
// so that it can start while the previous kernel of the stream drains.
//
// Until the previous kernel has finished, the CTA only warms L2 with the first
// weights of its range (an L2 prefetch cannot hide a later write).  Then warp
// CW, the producer, walks this CTA's output rows
// ("virtual rows" v; for FP4 v = i*N + n) in blocks of at most RB rows that
// never cross an expert boundary, and per block issues three bulk copies into
// a ring stage -- the block's packed rows (contiguous in the row-major
// matrix) and the 16-byte-aligned ranges enclosing its scale and zero rows --
// all completing on the stage's "full" mbarrier.  When a stage comes back it
// sums the consumers' per-warp partials of each row in a fixed order (results
// are bitwise reproducible) and writes the BF16 outputs.
//
// Warps 0..CW-1 consume.  They convert the activation once per CTA into
// shared memory (INT4: a 16-bit and an 8-bit integer part per value against a
// power-of-two scale per 128-element group, for exact dp2a / dp4a integer dot
// products; FP4: binary16 pairs with a scale per 32-element unit, for the
// mixed-precision FMA), then keep the part each thread owns in registers and
// work through the stages.
// All waits are bounded.
#pragma once

#include "common.cuh"
#include "gemv_common.cuh"
#include "kernels.h"

namespace w4 {

constexpr int kGemvMaxStages = 8;
constexpr int kGemvMaxRB = 32;
// Stages' worth of weights prefetched into L2 before the previous kernel
// ends: enough to start the stream at once, little enough not to queue the
// activation reads behind a burst of misses.
constexpr int kGemvPrefetchStages = 2;

struct GemvParams {
    const uint16_t *x;
    const uint8_t *qw;
    const uint16_t *s;
    const uint16_t *z;      // INT4 only; null: symmetric INT4 (zero point 8)
    const int32_t *ids;     // FP4 only
    uint16_t *y;
    unsigned int *status;
    int64_t rows_per_slot;  // FP4: N (one expert's rows); INT4: N
    int64_t V;              // virtual rows in total (INT4: N; FP4: topk * N)
    int64_t E;              // FP4: number of experts
    int64_t rows_q;         // V / grid (rows per CTA) ...
    int64_t rows_r;         // ... and V % grid (CTAs with one row more)
    int K, G, UPR, RB, stages;
    int64_t sz_total;       // bytes of the whole scale tensor (and of the zero tensor)
    int w_bytes;            // packed weights of a stage (RB * K/2)
    int sz_bytes;           // one scale (or zero) region of a stage, 16-aligned, with slack
    int x_off;              // byte offset of the converted activation (K/32 * 72 + 256 bytes)
    int stage_bytes;        // 128-aligned
    int stage_off;          // byte offset of stage 0
    unsigned int inject;    // test-only injection flags (0 normally)
    // batched decode (MV activation vectors, INT4 only), after the hot fields
    int64_t ldy;            // output row stride (N)
    int x_stride;           // bytes between the vectors' converted activations
    int mv_valid;           // vectors actually given (the rest are padding)
};

struct StageMeta {
    long long vrow;  // first virtual row of the block
    int rows;
    int valid;       // FP4: expert id in range
    int soff;        // half-words between the stage's s/z region start and the block's first group
    int pad;
};

template <int CW, int RPT>
struct GemvHeader {
    uint64_t full[kGemvMaxStages];
    uint64_t empty[kGemvMaxStages];
    StageMeta meta[kGemvMaxStages];
    float psum[kGemvMaxStages][2][CW][RPT];  // per-warp row partials, by phase parity
};


__device__ __forceinline__ int64_t gemv_even_floor(int64_t v) { return v & ~int64_t(1); }

template <bool FP4, int CW, int TT, int UPT, int RPT, bool SYM, int MV>
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
        if constexpr (MV == 1) {
            for (int r = lane; r < m.rows; r += 32) {
                const int team = r / RPT, rr = r - team * RPT;
                float acc = 0.0f;
#pragma unroll
                for (int w = 0; w < WPT; ++w) acc += h.psum[slot][par][team * WPT + w][rr];
                a.y[m.vrow + r] = m.valid ? f32_to_bf16_bits(acc) : static_cast<uint16_t>(0);
            }
        } else {
            // batched: vector v's rows were reduced by its own teams
            constexpr int TV = (CW * 32 / TT) / MV;  // teams per vector
            for (int idx = lane; idx < MV * m.rows; idx += 32) {
                const int vec = idx / m.rows, r = idx - vec * m.rows;
                if (vec >= a.mv_valid) continue;
                const int team = vec * TV + r / RPT, rr = r % RPT;
                float acc = 0.0f;
#pragma unroll
                for (int w = 0; w < WPT; ++w) acc += h.psum[slot][par][team * WPT + w][rr];
                a.y[vec * a.ldy + m.vrow + r] = f32_to_bf16_bits(acc);
            }
        }
    };
    int slot = 0, phase = 0, issued = 0;
    // After a wait ran out: wait (bounded, whatever the status word says)
    // until the copies of every stage issued and not yet retired have landed,
    // so that no copy into this CTA's shared memory is in flight when it
    // exits.  A stage's full barrier completes on its own copies alone.
    auto drain_copies = [&]() {
        const int first = issued > a.stages ? issued - a.stages : 0;
        for (int it = first; it < issued; ++it)
            mbar_wait(&h.full[it % a.stages], (it / a.stages) & 1, nullptr);
    };
    // Expert slot (FP4; INT4 has one slot of N rows) holding row `begin`.
    int64_t i_slot = FP4 ? begin / a.rows_per_slot : 0;
    int64_t slot_end = FP4 ? (i_slot + 1) * a.rows_per_slot : end;
    int64_t expert = FP4 && begin < end ? a.ids[i_slot] : 0;
    for (int64_t v = begin; v < end; ++issued) {
        const bool recycle = issued >= a.stages;
        StageMeta old{};
        if (recycle) {
            if (!mbar_wait(&h.empty[slot], phase ^ 1, a.status)) {
                drain_copies();
                return;
            }
            old = h.meta[slot];
            __syncwarp();
        }
        // The block: at most RB rows, not past this CTA's range nor the
        // current expert slot (no 64-bit division in this loop: a single
        // thread's division costs hundreds of nanoseconds here).
        int64_t lim = end - v;
        if (slot_end - v < lim) lim = slot_end - v;
        const int rows = static_cast<int>(lim < a.RB ? lim : a.RB);
        int64_t src_row = v;
        bool ok = true;
        if (FP4) {
            ok = (expert >= 0 && expert < a.E);
            src_row = (ok ? expert : 0) * a.rows_per_slot + (v - (slot_end - a.rows_per_slot));
        }
        unsigned char *st = stage0 + slot * a.stage_bytes;
        uint16_t *ss = reinterpret_cast<uint16_t *>(st + a.w_bytes);
        uint16_t *sz = reinterpret_cast<uint16_t *>(st + a.w_bytes + a.sz_bytes);
        // The block's scale (and zero) rows are one contiguous byte range
        // [b0, b1) of their tensor.  Its enclosing 16-byte-aligned chunks go
        // by 16-byte cp.async from the warp's lanes (keeping the bulk-copy
        // queue for the weights); a chunk that would pass the tensor's end
        // reads only the bytes before it and zero-fills the rest.
        const uint64_t b0 = static_cast<uint64_t>(src_row) * a.G * 2;
        const uint64_t b1 = b0 + static_cast<uint64_t>(rows) * a.G * 2;
        const uint64_t lo16 = b0 & ~uint64_t(15);
        if (lane == 0) {
            if (!ok) atomicOr(a.status, kDevBadExpert);
            h.meta[slot].vrow = v;
            h.meta[slot].rows = rows;
            h.meta[slot].valid = ok ? 1 : 0;
            h.meta[slot].soff = static_cast<int>((b0 - lo16) >> 1);
            const uint32_t wb = ok ? static_cast<uint32_t>(rows) * half_k : 0u;
            mbar_arrive_expect_tx(&h.full[slot], wb);
            if (ok) bulk_g2s(st, a.qw + src_row * half_k, wb, &h.full[slot], pol);
        }
        if (ok) {
            const unsigned char *gs = reinterpret_cast<const unsigned char *>(a.s);
            const unsigned char *gz = reinterpret_cast<const unsigned char *>(a.z);
            for (uint64_t o = lo16 + 16 * static_cast<uint64_t>(lane); o < b1; o += 16 * 32) {
                const uint64_t left = static_cast<uint64_t>(a.sz_total) - o;
                const uint32_t n = left < 16 ? static_cast<uint32_t>(left) : 16u;
                cp_async_16_zfill(reinterpret_cast<unsigned char *>(ss) + (o - lo16), gs + o, n);
                if (!FP4 && !SYM) cp_async_16_zfill(reinterpret_cast<unsigned char *>(sz) + (o - lo16), gz + o, n);
            }
        }
        cp_async_arrive_noinc(&h.full[slot]);
        // the next copy is in flight; now finish the block this slot held
        if (recycle) finalize(slot, phase ^ 1, old);
        v += rows;
        if (FP4 && v == slot_end && v < end) {
            ++i_slot;
            slot_end += a.rows_per_slot;
            expert = a.ids[i_slot];
        }
        if (++slot == a.stages) {
            slot = 0;
            phase ^= 1;
        }
    }
    // drain: finish the last min(stages, issued) blocks
    const int first = issued > a.stages ? issued - a.stages : 0;
    for (int it = first; it < issued; ++it) {
        const int sl = it % a.stages;
        if (!mbar_wait(&h.empty[sl], (it / a.stages) & 1, a.status)) {
            drain_copies();
            return;
        }
        finalize(sl, (it / a.stages) & 1, h.meta[sl]);
    }
}

// L2 prefetch of the first kGemvPrefetchStages blocks of this CTA's range:
// the packed codes by bulk prefetch (from the producer lane, ahead of its own
// stage copies), the scale and zero rows one 32-byte sector per instruction
// from the consumer threads (idle until the previous kernel ends).  Ranges
// are rounded inward to 16 bytes, so no address leaves its tensor.
__device__ __forceinline__ int64_t gemv_prefetch_rows(const GemvParams &a, int64_t begin, int64_t end) {
    int64_t rows = static_cast<int64_t>(kGemvPrefetchStages) * a.RB;
    return rows < end - begin ? rows : end - begin;
}

__device__ __forceinline__ void gemv_prefetch_codes(const GemvParams &a, int64_t begin, int64_t end) {
    const int64_t rows = gemv_prefetch_rows(a, begin, end);
    const int64_t half_k = a.K >> 1;
    const unsigned char *p = a.qw + begin * half_k;
    for (int64_t o = 0; o < rows * half_k; o += 32768) {
        const int64_t n = rows * half_k - o < 32768 ? rows * half_k - o : 32768;
        prefetch_l2_bulk(p + o, static_cast<uint32_t>(n));  // half_k % 64 == 0: aligned, whole
    }
}

__device__ __forceinline__ void gemv_prefetch_range(const void *base, uint64_t lo, uint64_t hi, int tid,
                                                    int nthreads) {
    lo = (lo + 15) & ~uint64_t(15);
    hi &= ~uint64_t(15);
    const unsigned char *p = static_cast<const unsigned char *>(base);
    for (uint64_t o = lo + static_cast<uint64_t>(tid) * 32; o < hi; o += static_cast<uint64_t>(nthreads) * 32)
        prefetch_l2_line(p + o);
}

template <bool SYM>
__device__ __forceinline__ void gemv_prefetch_groups(const GemvParams &a, int64_t begin, int64_t end, int tid,
                                                     int nthreads) {
    const int64_t rows = gemv_prefetch_rows(a, begin, end);
    const uint64_t g0 = static_cast<uint64_t>(begin) * a.G * 2, g1 = static_cast<uint64_t>(begin + rows) * a.G * 2;
    gemv_prefetch_range(a.s, g0, g1, tid, nthreads);
    if (!SYM) gemv_prefetch_range(a.z, g0, g1, tid, nthreads);
}

// Activation conversion, once per CTA, into shared memory at xs, laid out as
// uint4 "planes" so that the threads' later register loads are free of bank
// conflicts.
//  INT4: one 32-value unit per thread (K/32 units; the four units of a group
//        are four neighbouring lanes, K % 128 == 0 keeps every group whole).
//        Plane p = 4s + i (s: 32-value unit within the group, i: word within
//        the unit) holds Gp = G rounded up to even entries, one per group;
//        plane 16 holds per group (sum of hi, set-aside list, x of the first
//        and of the second set-aside value), the list packing their
//        positions in the group (bits 0-6, 8-14), their count (bits 16-17)
//        and e + 128 (bits 24-31).
//  FP4:  one 32-value unit per thread; plane i holds U = K/32 entries, one
//        per unit; per unit a float2 (0, pw) at xs + 64U + 256.
__device__ __forceinline__ int gemv_x_consts(int K) { return (K >> 5) * 64 + 256; }
__device__ __host__ __forceinline__ int gemv_x_gp(int K) { return ((K >> 7) + 1) & ~1; }
__device__ __host__ __forceinline__ int gemv_int4_x_bytes(int K) { return 17 * 16 * gemv_x_gp(K); }

// FP4: one 32-value unit u of activation x into the planes at xs; `ok`
// false: a padding lane, which stores nothing.
__device__ __forceinline__ void gemv_convert_fp4_unit(const uint16_t *x, unsigned char *xs, int u, bool ok,
                                                      int units) {
    uint4 *xw = reinterpret_cast<uint4 *>(xs);
    uint32_t xb[16], w[16];
    if (ok) {
        load_x_unit(x + 32 * u, xb);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) xb[i] = 0u;
    }
    const float2 c = make_float2(0.0f, fp4_x_unit(xb, w));
    if (ok) {
#pragma unroll
        for (int i = 0; i < 4; ++i) xw[i * units + u] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        reinterpret_cast<float2 *>(xs + gemv_x_consts(units * 32))[u] = c;
    }
}

// INT4: one 32-value unit u (= 4 words) of an activation of K values into
// the planes at xs (the layout above).  The four units of a group are four
// neighbouring lanes; all 32 lanes of the warp call it together (the group
// shuffles); `ok` false: a padding lane (of a whole padding group), which
// stores nothing.  CG: load through L2 only (in a chain of linears the
// activation may have been written by another CTA of the same launch).
template <bool CG>
__device__ __forceinline__ void gemv_convert_int4_unit(const uint16_t *x, unsigned char *xs, int u, bool ok, int K) {
    uint4 *xw = reinterpret_cast<uint4 *>(xs);
    const int lane = threadIdx.x & 31;
    uint32_t xb[16];
    if (ok) {
        const uint4 *p = reinterpret_cast<const uint4 *>(x + 32 * u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = CG ? __ldcg(p + q) : p[q];
            xb[4 * q] = v.x;
            xb[4 * q + 1] = v.y;
            xb[4 * q + 2] = v.z;
            xb[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) xb[i] = 0u;
    }
    // the group's largest |x| (exponent e1) and how many values have an
    // exponent of at least e1 - 1
    uint32_t m = unit_absmax_bits(xb);
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    int e = exponent_of_absmax(m);
    int c = (m & 0x7F80u) > 0x0080u ? count_at_least<16>(xb, (m & 0x7F80u) - 0x0080u) : 3;
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    Top3 t = {0u, 0u, 0u, 0u, 0u, 0u, 0u};
    bool o1 = false, o2 = false;
    // the third largest more than one binade below the largest: the largest
    // one or two may lie above the third largest's binade (warp-uniform
    // branch: the group search shuffles)
    if (__any_sync(0xffffffffu, c < 3)) {
        t = group_top3<4>(xb, lane);
        if (c < 3) {
            const bool few = t.a3 == 0u;  // at most two nonzero values: set them aside
            e = few ? 0 : exponent_of_absmax(t.a3);
            const uint32_t thr = static_cast<uint32_t>(e + 128) << 7;  // magnitude bits of 2^(e+1)
            o1 = t.a1 != 0u && (few || t.a1 >= thr);
            o2 = t.a2 != 0u && (few || t.a2 >= thr);  // implies o1
        }
    }
    uint32_t w[16];
    uint32_t usum = int4_x_unit(xb, e, w);
    // the set-aside values among this lane's 32: out of the integer part
    const uint32_t mine = static_cast<uint32_t>(u & 3);
    if (__any_sync(0xffffffffu, o1)) {  // rare: keep the common path free of it
        usum -= int4_x_drop(w, xb, o1 && (t.p1 >> 5) == mine ? t.p1 & 31u : 32u, e);
        usum -= int4_x_drop(w, xb, o2 && (t.p2 >> 5) == mine ? t.p2 & 31u : 32u, e);
    }
    int sum = static_cast<int>(usum);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (ok) {
        const int gp = gemv_x_gp(K), grp = u >> 2, sub = u & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            xw[(4 * sub + i) * gp + grp] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        if (sub == 0) {
            const uint32_t n = (o1 ? 1u : 0u) + (o2 ? 1u : 0u);
            const uint32_t list = (o1 ? t.p1 : 0u) | ((o2 ? t.p2 : 0u) << 8) | (n << 16) |
                                  (static_cast<uint32_t>(e + 128) << 24);
            // |sum| <= 128 * 32640 < 2^23: exact in binary32
            xw[16 * gp + grp] = make_uint4(__float_as_uint(static_cast<float>(sum)), list,
                                           __float_as_uint(bf16_bits_to_f32(t.v1)),
                                           __float_as_uint(bf16_bits_to_f32(t.v2)));
        }
    }
}

// The whole activation x (K values) by consumer warps warp, warp + nwarps,
// ..., one 32-value unit a thread.  Every CTA reads the same few KB at the
// same moment; starting each CTA at a different group (a rotation by whole
// groups) spreads the requests over the L2 slices.
template <bool FP4, bool CG = false>
__device__ __forceinline__ void gemv_convert_vector(const uint16_t *x, unsigned char *xs, int K, int warp, int nwarps,
                                                    int lane) {
    const int units = K >> 5;
    if constexpr (FP4) {
        const int rot = static_cast<int>((blockIdx.x * 7u) % static_cast<unsigned>(units));
        for (int u0 = warp * 32; u0 < units; u0 += nwarps * 32) {  // warp-uniform
            const bool ok = u0 + lane < units;
            int u = u0 + lane + rot;
            if (u >= units) u -= units;
            gemv_convert_fp4_unit(x, xs, u, ok, units);
        }
    } else {
        const int rot = 4 * static_cast<int>((blockIdx.x * 7u) % static_cast<unsigned>(units >> 2));
        for (int u0 = warp * 32; u0 < units; u0 += nwarps * 32) {  // warp-uniform
            const bool ok = u0 + lane < units;                     // the four lanes of a group share ok
            int u = u0 + lane + rot;
            if (u >= units) u -= units;
            gemv_convert_int4_unit<CG>(x, xs, u, ok, K);
        }
    }
}

// A consumer thread's INT4 activation: its group's 64 words of hi pairs (four
// sub-units, in the thread's rotated order) and constants.
struct Int4X {
    uint32_t xh[4][16];
    float sum;
    float pw;  // 2^(e-14), negated when the group has set-aside values (their list stays in shared memory)
};

__device__ __forceinline__ void int4_load_x(const unsigned char *xs, int gp, int gs, int rot, bool valid, Int4X &r) {
    const uint4 *xw = reinterpret_cast<const uint4 *>(xs);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int sub = (q + rot) & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v4 = xw[(4 * sub + i) * gp + gs];
            r.xh[q][4 * i] = v4.x;
            r.xh[q][4 * i + 1] = v4.y;
            r.xh[q][4 * i + 2] = v4.z;
            r.xh[q][4 * i + 3] = v4.w;
        }
    }
    const uint4 c = xw[16 * gp + gs];
    r.sum = __uint_as_float(c.x);
    const float pw = valid ? pow2f(static_cast<int>(c.y >> 24) - 128 - 14) : 0.0f;
    r.pw = (valid && ((c.y >> 16) & 3u)) ? -pw : pw;
}

// One stage's work of a consumer thread: RPT rows (from rbase) of its group
// g; codes at st + row * half_k + 64 g, the 16-byte sub-units taken in
// rotated order; ss / sz: the stage's scale and zero rows (sz unused when
// sym); xc: the group's plane-16 entry.  Adds each row's contribution to
// part[].
template <int RPT>
__device__ __forceinline__ void int4_group_rows(const Int4X &x, const unsigned char *st, int half_k, int rbase, int g,
                                                int rot, const uint16_t *ss, const uint16_t *sz, bool sym, int G,
                                                const uint4 *xc, float (&part)[RPT]) {
    int lo[RPT], hi[RPT];
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) lo[rr] = hi[rr] = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int sub = (q + rot) & 3;
        uint4 wv[RPT];
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr)
            wv[rr] = *reinterpret_cast<const uint4 *>(st + static_cast<size_t>(rbase + rr) * half_k + 64 * g + 16 * sub);
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr) {
            const uint32_t words[4] = {wv[rr].x, wv[rr].y, wv[rr].z, wv[rr].w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                // even codes as bytes c (one logic op), odd codes as bytes
                // 16c (one logic op, no shift)
                const uint32_t ev = words[m] & 0x0F0F0F0Fu, od = words[m] & 0xF0F0F0F0u;
                lo[rr] = dp2a_lo(x.xh[q][4 * m + 0], ev, lo[rr]);
                lo[rr] = dp2a_hi(x.xh[q][4 * m + 1], ev, lo[rr]);
                hi[rr] = dp2a_lo(x.xh[q][4 * m + 2], od, hi[rr]);
                hi[rr] = dp2a_hi(x.xh[q][4 * m + 3], od, hi[rr]);
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
        // hi is a multiple of 16 (exact shift); |dot| < 2^26 (the conversion
        // to binary32 rounds it by at most 2^-24 of itself)
        const int dot = lo[rr] + (hi[rr] >> 4);
        const int gi = (rbase + rr) * G + g;
        const float sv = f16_bits_to_f32(ss[gi]);
        const float zf = sym ? 8.0f : f16_bits_to_f32(sz[gi]);  // symmetric: the midpoint 8
        float acc = (sv * fabsf(x.pw)) * fmaf(-zf, x.sum, static_cast<float>(dot));
        if (x.pw < 0.0f) {
            // the set-aside values: s (q - z) x, each product exact in binary32
            // (the activation region is not rewritten while the rows run)
            const unsigned char *row = st + static_cast<size_t>(rbase + rr) * half_k + 64 * g;
            const uint4 c = *xc;
            const uint32_t n = (c.y >> 16) & 3u;
            const uint32_t p1 = c.y & 127u;
            const float c1 = static_cast<float>((row[p1 >> 1] >> ((p1 & 1u) * 4u)) & 15u);
            acc = fmaf(sv * (c1 - zf), __uint_as_float(c.z), acc);
            if (n > 1) {
                const uint32_t p2 = (c.y >> 8) & 127u;
                const float c2 = static_cast<float>((row[p2 >> 1] >> ((p2 & 1u) * 4u)) & 15u);
                acc = fmaf(sv * (c2 - zf), __uint_as_float(c.w), acc);
            }
        }
        part[rr] += acc;
    }
}

// The activation (MV == 1), or the MV activation vectors x0 + v K of a
// batched pass (padding vectors, v >= a.mv_valid, repeat the last given one),
// vector v into xs0 + v * x_stride.
template <bool FP4, int CW, int MV>
__device__ __forceinline__ void gemv_convert_x(const GemvParams &a, const uint16_t *x0, unsigned char *xs0, int warp,
                                               int lane) {
    if constexpr (MV == 1) {
        gemv_convert_vector<FP4>(x0, xs0, a.K, warp, CW, lane);
    } else {
#pragma unroll 1
        for (int v = 0; v < MV; ++v)
            gemv_convert_vector<FP4>(x0 + static_cast<int64_t>(min(v, a.mv_valid - 1)) * a.K, xs0 + v * a.x_stride,
                                     a.K, warp, CW, lane);
    }
}

// After a stage: reduce the per-row partials across the warp, park them for
// the producer and release the stage.
template <int CW, int RPT>
__device__ __forceinline__ void gemv_release_stage(GemvHeader<CW, RPT> &h, const float (&part)[RPT], int slot,
                                                   int phase, int warp, int lane) {
    const float red = warp_reduce_rows<RPT>(part, lane);
    if ((lane & (32 / RPT - 1)) == 0) h.psum[slot][phase][warp][reduced_row<RPT>(lane)] = red;
    __syncwarp();
    if (lane == 0) mbar_arrive(&h.empty[slot]);
}

// INT4 consumer.  A thread owns one 128-code group g of RPT rows per stage:
// 64 bytes of packed codes per row, read as four 16-byte sub-units (u = 4g+s).
// Lanes start at different sub-units (rotation (g >> 1) & 3) so that the
// eight lanes of each 128-byte shared-memory wavefront hit distinct banks;
// the x registers are loaded in the same rotated order, so indexing stays
// static.  Products are exact integer dot products (dp2a); per (row, group):
//   y += s * 2^(e-14) * (dot - z * sum_hi) + sum over set-aside x of s * (q - z) * x.
template <int CW, int TT, int RPT, bool SYM, int MV>
__device__ __forceinline__ void gemv_consume_int4(const GemvParams &a, GemvHeader<CW, RPT> &h,
                                                  const unsigned char *stage0, const unsigned char *xs0,
                                                  int64_t begin, int64_t end, int warp, int lane) {
    // batched (MV > 1): the teams split into MV sets, one per activation
    // vector, each set covering every row of a stage
    constexpr int TV = (CW * 32 / TT) / MV;  // teams per vector
    const int team0 = threadIdx.x / TT;
    const int vec = MV == 1 ? 0 : team0 / TV;
    const int team = MV == 1 ? team0 : team0 % TV;
    const unsigned char *xs = MV == 1 ? xs0 : xs0 + vec * a.x_stride;
    const int g = threadIdx.x % TT;
    const bool valid = g < a.G;
    const int gs = valid ? g : 0;
    const int rot = (g >> 1) & 3;
    Int4X x;
    int4_load_x(xs, gemv_x_gp(a.K), gs, rot, valid, x);
    const int half_k = a.K >> 1;

    const int rbase = team * RPT;
    int slot = 0, phase = 0;
    for (int64_t v = begin; v < end;) {
        if (!mbar_wait(&h.full[slot], phase, a.status)) return;
        const int rows = h.meta[slot].rows;
        const int soff = h.meta[slot].soff;
        const unsigned char *st = stage0 + slot * a.stage_bytes;
        const uint16_t *ss = reinterpret_cast<const uint16_t *>(st + a.w_bytes) + soff;
        const uint16_t *sz = reinterpret_cast<const uint16_t *>(st + a.w_bytes + a.sz_bytes) + soff;
        float part[RPT];
#pragma unroll
        for (int rr = 0; rr < RPT; ++rr) part[rr] = 0.0f;
        if (valid)
            int4_group_rows<RPT>(x, st, half_k, rbase, gs, rot, ss, sz, SYM, a.G,
                                 reinterpret_cast<const uint4 *>(xs) + 16 * gemv_x_gp(a.K) + gs, part);
        gemv_release_stage<CW, RPT>(h, part, slot, phase, warp, lane);
        v += rows;
        if (++slot == a.stages) {
            slot = 0;
            phase ^= 1;
        }
    }
}

// FP4 consumer.  A thread owns UPT 32-code units (u = j + i*TT) of RPT rows
// per stage; codes decode exactly to binary16 pairs (cvt e2m1x2) and meet the
// f16 activation pairs in the mixed-precision FMA; one scale per unit.
template <int CW, int TT, int UPT, int RPT>
__device__ __forceinline__ void gemv_consume_fp4(const GemvParams &a, GemvHeader<CW, RPT> &h,
                                                 const unsigned char *stage0, const unsigned char *xs,
                                                 int64_t begin, int64_t end, int warp, int lane) {
    const int team = threadIdx.x / TT;
    const int j = threadIdx.x % TT;
    const int units = a.K >> 5;
    const uint4 *xw = reinterpret_cast<const uint4 *>(xs);
    const float2 *xc = reinterpret_cast<const float2 *>(xs + gemv_x_consts(a.K));
    uint32_t xr[UPT][16];
    float pw[UPT];
    bool valid[UPT];
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
        const int u = j + i * TT;
        valid[i] = u < units;
        const int us = valid[i] ? u : 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v4 = xw[q * units + us];
            xr[i][4 * q] = v4.x;
            xr[i][4 * q + 1] = v4.y;
            xr[i][4 * q + 2] = v4.z;
            xr[i][4 * q + 3] = v4.w;
        }
        pw[i] = valid[i] ? xc[us].y : 0.0f;
    }

    const int rbase = team * RPT;
    int slot = 0, phase = 0;
    for (int64_t v = begin; v < end;) {
        if (!mbar_wait(&h.full[slot], phase, a.status)) return;
        const int rows = h.meta[slot].rows;
        const int soff = h.meta[slot].soff;
        const unsigned char *st = stage0 + slot * a.stage_bytes;
        const uint16_t *ss = reinterpret_cast<const uint16_t *>(st + a.w_bytes) + soff;
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
                wv[rr] = *reinterpret_cast<const uint4 *>(st + (static_cast<size_t>(rbase + rr) * units + u) * 16);
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr) {
                const uint32_t words[4] = {wv[rr].x, wv[rr].y, wv[rr].z, wv[rr].w};
                float lo = 0.0f, hi = 0.0f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint32_t h[4];
                    e2m1x8_to_f16x2(words[m], h);
#pragma unroll
                    for (int b = 0; b < 4; ++b) mfma_f16x2(h[b], xr[i][4 * m + b], lo, hi);
                }
                const float sf = f16_bits_to_f32(ss[(rbase + rr) * a.G + u]) * pw[i];
                part[rr] = fmaf(sf, lo + hi, part[rr]);
            }
        }
        gemv_release_stage<CW, RPT>(h, part, slot, phase, warp, lane);
        v += rows;
        if (++slot == a.stages) {
            slot = 0;
            phase ^= 1;
        }
    }
}

template <bool FP4, int CW, int TT, int UPT, int RPT, bool SYM, int MV>
__global__ void __launch_bounds__((CW + 1) * 32, 1) gemv_stream_kernel(const GemvParams a) {
    using Header = GemvHeader<CW, RPT>;
    extern __shared__ __align__(1024) unsigned char smem[];
    Header &h = *reinterpret_cast<Header *>(smem);
    unsigned char *stage0 = smem + a.stage_off;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // This CTA's contiguous range of virtual rows: V = q * grid + r rows,
    // the first r CTAs take one more (q and r come from the host).
    const int64_t b = blockIdx.x;
    const int64_t begin = b * a.rows_q + (b < a.rows_r ? b : a.rows_r);
    const int64_t end = begin + a.rows_q + (b < a.rows_r ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&h.full[i], 33);  // producer lane 0 (+ weight bytes) and its 32 cp.async lanes
            mbar_init(&h.empty[i], CW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // The next launch of the stream may now be scheduled: its CTAs take the
    // SMs this grid frees and warm L2 with their first weights while this
    // grid drains.
    pdl_launch_dependents();

    if (warp == CW) {
        if (!FP4 && lane == 0) gemv_prefetch_codes(a, begin, end);
        // The weights copied into shared memory, the expert ids and the
        // output follow the stream order.
        pdl_wait();
        // test-only injection: no stage is ever issued, so the consumers'
        // first waits run out and the launch ends with the timeout status
        if (!(a.inject & kInjectStallPipeline))
            gemv_producer<FP4, CW, TT, UPT, RPT, SYM, MV>(a, h, stage0, begin, end, lane);
        return;
    }

    // Until the previous kernel ends only the L2 prefetch of this CTA's first
    // weights may run (it cannot hide a later write: L2 is the point of
    // coherence).  The activation follows the stream order: the consumers
    // convert it once per CTA into shared memory, then each thread copies the
    // part it owns into registers.
    if (!FP4) gemv_prefetch_groups<SYM>(a, begin, end, threadIdx.x, CW * 32);
    pdl_wait();
    // test-only injection: the consumers take no stage, so the producer's
    // waits for free stages run out with its copies issued
    if (a.inject & kInjectStallConsumers) return;
    gemv_convert_x<FP4, CW, MV>(a, a.x, smem + a.x_off, warp, lane);
    named_bar_sync(1, CW * 32);
    if constexpr (FP4)
        gemv_consume_fp4<CW, TT, UPT, RPT>(a, h, stage0, smem + a.x_off, begin, end, warp, lane);
    else
        gemv_consume_int4<CW, TT, RPT, SYM, MV>(a, h, stage0, smem + a.x_off, begin, end, warp, lane);
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
    // Four rows per thread whenever the block fits: more independent work per
    // stage hand-off (measured: 64 experts of 4096 x 7168, top 6 -- 24.9 us
    // against 29.8 us with two rows and stages kept under the stage target).
    const int teams = CW * 32 / best.TT;
    best.RPT = (teams * 4 <= kGemvMaxRB) ? 4 : 2;
    (void)row_bytes;
    (void)stage_target;
    return best;
}

constexpr int kGemvCW = 16;             // consumer warps per CTA

// Teams of an INT4 CTA at this K: the activation vectors one pass carries
// (MV) split the teams into one set per vector, so MV must divide this.
inline int gemv_int4_teams(int64_t K) {
    int tt = 32;
    while (tt < K / 128) tt *= 2;
    return kGemvCW * 32 / tt;
}
constexpr int kGemvStageTarget = 32768; // packed weight bytes per stage (upper aim)
constexpr int kGemvShortRing = 4;        // ring depth for a CTA share of ...
constexpr int kGemvShortShareStages = 8; // ... at most this many stages of weights

template <bool FP4, int TT, int UPT, int RPT, bool SYM, int MV = 1>
cudaError_t gemv_launch(GemvParams a, cudaStream_t st, int device, int num_sms, int max_smem) {
    constexpr int CW = kGemvCW;
    auto kern = gemv_stream_kernel<FP4, CW, TT, UPT, RPT, SYM, MV>;
    const int header = (static_cast<int>(sizeof(GemvHeader<CW, RPT>)) + 127) & ~127;
    a.x_off = header;
    // converted x per vector (a multiple of 16): FP4 planes, then (0, pw) per
    // unit; INT4 hi and lo planes, then the per-half-group constants
    a.x_stride = FP4 ? (a.K / 32) * 72 + 256 : gemv_int4_x_bytes(a.K);
    a.stage_off = (a.x_off + MV * a.x_stride + 1023) & ~1023;
    int64_t ctas = num_sms;
    const int64_t max_ctas = (a.V + 1) / 2;  // at least two rows each
    if (ctas > max_ctas) ctas = max_ctas;
    if (ctas < 1) ctas = 1;
    int stages = (max_smem - a.stage_off) / a.stage_bytes;
    if (stages > kGemvMaxStages) stages = kGemvMaxStages;
    // A CTA whose whole share of the weights fits in a few stages gets a
    // ring of kGemvShortRing: the later stages are then requested as the
    // first ones are consumed rather than all at once (measured, decode MLP
    // pair 15360 x 3840 then 3840 x 15360: 14.95 against 15.19 us per pair
    // with 7 stages).  Longer shares keep the deepest ring (the 262144 x
    // 3840 vocabulary GEMV: 73.2 us with 7, 74.5 with 4).
    const int64_t share = (a.V + ctas - 1) / ctas * static_cast<int64_t>(a.K / 2);
    if (share <= kGemvShortShareStages * static_cast<int64_t>(a.stage_bytes) && stages > kGemvShortRing)
        stages = kGemvShortRing;
    if (stages < 2) return cudaErrorInvalidValue;
    a.stages = stages;
    const int smem = a.stage_off + stages * a.stage_bytes;
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure(reinterpret_cast<const void *>(kern), device, smem)) return e;
    a.rows_q = a.V / ctas;
    a.rows_r = a.V % ctas;
    // Programmatic stream serialisation: this launch may begin while the
    // previous kernel of the stream finishes; the kernel waits for it
    // (griddepcontrol.wait) before touching x, y or the expert ids.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3((CW + 1) * 32);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Fill the stage geometry of `a` for K and launch the matching instance.
//  INT4: a thread owns one 128-code group: TT = the smallest power-of-two
//        warp multiple covering K/128 groups; RPT = 2 rows per thread while a
//        stage stays within the stage target, else 1.
//  FP4:  TT threads x UPT units of 32 codes cover a row (gemv_choose_shape).
// SYM: symmetric INT4 (no zero points), its own kernel instances so that the
// asymmetric ones carry no test for it.  MV > 1 (INT4): MV activation vectors
// share one pass over the weights; each thread then takes MV rows per stage
// (RPT = MV) and a stage holds one row per team.
template <bool FP4, bool SYM = false, int MV = 1>
cudaError_t gemv_dispatch(GemvParams a, cudaStream_t st, int device, int num_sms, int max_smem) {
    static_assert(MV == 1 || !FP4, "batched vectors: INT4 only");
    const int row_bytes = a.K / 2;
    GemvShape sh = {0, 0, 0};
    if (FP4) {
        a.UPR = a.K / 32;
        sh = gemv_choose_shape(kGemvCW, a.UPR, row_bytes, kGemvStageTarget);
    } else {
        a.UPR = a.G;  // groups per row, one per thread
        for (int tt = 32; tt <= 128 && sh.TT == 0; tt *= 2)
            if (tt >= a.G) sh = {tt, 1, 0};
        if (sh.TT != 0) {
            const int teams = kGemvCW * 32 / sh.TT;
            if (MV > 1) {
                if (teams % MV != 0) return cudaErrorInvalidValue;
                sh.RPT = MV;
            } else {
                sh.RPT = (teams * 2 * row_bytes <= kGemvStageTarget && teams * 2 <= kGemvMaxRB) ? 2 : 1;
            }
        }
    }
    if (sh.TT == 0) return cudaErrorInvalidValue;
    a.RB = (kGemvCW * 32 / sh.TT) * sh.RPT / MV;
    if (a.RB > kGemvMaxRB) return cudaErrorInvalidValue;
    a.w_bytes = a.RB * row_bytes;
    a.sz_bytes = ((a.RB * a.G * 2) + 32 + 15) & ~15;  // + slack for the 16-byte-aligned superset
    a.stage_bytes = (a.w_bytes + (FP4 ? 1 : 2) * a.sz_bytes + 127) & ~127;
    if constexpr (FP4) {
#define W4_GEMV_CASE(TT_, UPT_)                                                                   \
    if (sh.TT == TT_ && sh.UPT == UPT_)                                                           \
        return sh.RPT == 4 ? gemv_launch<true, TT_, UPT_, 4, false>(a, st, device, num_sms, max_smem) \
                           : gemv_launch<true, TT_, UPT_, 2, false>(a, st, device, num_sms, max_smem);
        W4_GEMV_CASE(32, 2)
        W4_GEMV_CASE(64, 2)
        W4_GEMV_CASE(128, 2)
        W4_GEMV_CASE(256, 2)
        W4_GEMV_CASE(32, 1)
#undef W4_GEMV_CASE
    } else if constexpr (MV == 1) {
#define W4_GEMV_CASE(TT_)                                                                         \
    if (sh.TT == TT_)                                                                             \
        return sh.RPT == 2 ? gemv_launch<false, TT_, 1, 2, SYM>(a, st, device, num_sms, max_smem) \
                           : gemv_launch<false, TT_, 1, 1, SYM>(a, st, device, num_sms, max_smem);
        W4_GEMV_CASE(32)
        W4_GEMV_CASE(64)
        W4_GEMV_CASE(128)
#undef W4_GEMV_CASE
    } else {
        if (sh.TT == 32) return gemv_launch<false, 32, 1, MV, SYM, MV>(a, st, device, num_sms, max_smem);
        if (sh.TT == 64) return gemv_launch<false, 64, 1, MV, SYM, MV>(a, st, device, num_sms, max_smem);
        if (sh.TT == 128) return gemv_launch<false, 128, 1, MV, SYM, MV>(a, st, device, num_sms, max_smem);
    }
    return cudaErrorInvalidValue;
}

}  // namespace w4
