// Shared device helpers for the sm_103a kernels: inline-PTX wrappers for
// mbarriers, bulk asynchronous copies, and the sticky device status word.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace w4 {

// Bits of the per-device status word written by kernels (never by traps).
enum : unsigned int {
    kDevTimeout = 1u,    // a pipeline wait exceeded its time limit
    kDevBadExpert = 2u,  // an expert id outside [0, E)
};
// Test-only injection flags, passed to the kernels as an argument: with
// kInjectStallPipeline the producers issue nothing, so that the waits on
// them run out; with kInjectStallConsumers the consumers take nothing, so
// that the producers' waits run out while their copies are issued -- the
// bounded-wait paths, exercised without a fault.
enum : unsigned int {
    kInjectStallPipeline = 1u,
    kInjectStallConsumers = 2u,
};

// Wait limit for every mbarrier spin, in nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Make barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], "
        "%1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread may sleep up to hint_ns
// (woken when the phase completes) instead of returning after the default
// short time slice, so a waiting warp leaves its issue slots to the others.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

template <uint32_t HINT>
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
    return HINT ? mbar_try_wait_hint(bar, parity, HINT) : mbar_try_wait(bar, parity);
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false (and records kDevTimeout) if it did not complete within the limit, or
// at once if some wait of this device already timed out, so that a failing
// launch winds down quickly instead of sitting out one limit per wait.
// A barrier check is a dependent shared-memory round trip of roughly 150 SM
// cycles even when the phase has completed, so the common case is a single
// try_wait ahead of the loop.
// HINT (ns, 0: none) is the suspend-time hint of the polls after the first.
template <uint32_t HINT = 0>
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          unsigned int *status) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    // try_wait suspends the thread until the phase completes or a short
    // hardware time slice ends, so polling it costs no memory traffic; the
    // clock and the status word are consulted only between batches.
#pragma unroll 1
    for (int i = 0; i < 1024; ++i)
        if (mbar_poll<HINT>(a, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
#pragma unroll 1
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 1024; ++i)
            if (mbar_poll<HINT>(a, parity)) return true;
        if (status && (*reinterpret_cast<volatile unsigned int *>(status) & kDevTimeout)) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            if (status) atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// Warp-wide bounded wait on up to 32 barriers at once: each lane names its
// own barrier (or none, bar == nullptr) and parity, and every lane returns
// once all of them have completed -- one barrier round trip for the whole
// set instead of one per barrier.  All 32 lanes must call it together.
// Returns false on timeout (every lane alike).
template <uint32_t HINT = 0>
__device__ __forceinline__ bool mbar_wait_lanes(uint64_t *bar, uint32_t parity, unsigned int *status) {
    const uint32_t a = bar ? smem_u32(bar) : 0u;
    bool done = (bar == nullptr) || mbar_try_wait(a, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    const unsigned long long t0 = global_timer_ns();
#pragma unroll 1
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 256; ++i) {
            if (!done) done = mbar_poll<HINT>(a, parity);
            if (__all_sync(0xffffffffu, done)) return true;
        }
        const bool stop = (status && (*reinterpret_cast<volatile unsigned int *>(status) & kDevTimeout)) ||
                          global_timer_ns() - t0 > kWaitLimitNs;
        if (__any_sync(0xffffffffu, stop)) {
            if (status && (threadIdx.x & 31) == 0) atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// L2 policy: the packed weights are streamed exactly once.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
                 : "=l"(p));
    return p;
}

// L2 policy for small operands that every CTA reads (the activation).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// One-dimensional bulk copy global -> this CTA's shared memory, completing
// `bytes` transaction bytes on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src,
                                         uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes."
        "L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (no destination, no barrier);
// src 16-byte aligned, bytes % 16 == 0.  L2 is the point of coherence, so a
// prefetched line never hides a later write by another kernel.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Prefetch the 128-byte line holding p into L2 (through the load/store unit,
// not the bulk-copy engine).
__device__ __forceinline__ void prefetch_l2_line(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of
// the stream (launched with programmatic stream serialisation) be scheduled
// before this grid ends; wait blocks the calling thread until every grid this
// one depends on has completed and its memory operations are visible.  Both
// are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Four-byte asynchronous copy global -> shared (LDGSTS), 4-byte aligned.
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
                 "l"(src)
                 : "memory");
}

// Sixteen-byte asynchronous copy global -> shared that bypasses L1; only the
// first `src_bytes` (0 or 16) are read, the rest of the 16 bytes are zeros.
__device__ __forceinline__ void cp_async_16_zfill(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Arrive on `bar` once all of this thread's earlier cp.async copies land;
// the arrival counts toward the barrier's expected count.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) {
    return __uint_as_float(b << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t b) {
    return __half2float(__ushort_as_half(b));
}

}  // namespace w4
