// C ABI (include/w4a16.h): argument checks on the host, then one launch.
// Nothing here allocates device memory or synchronises except
// w4a16_check_device_error, which synchronises the given stream by design.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <new>

#include "w4a16.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// Sticky per-device status word (bits in common.cuh).  A __device__ variable
// exists once per device context; its address is looked up per device at
// first use.
__device__ unsigned int g_status;

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return W4A16_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device state, filled once per device under a mutex (host threads may
// make their first calls concurrently); after that it is read without a lock.
struct DevCache {
    std::atomic<bool> ready{false};
    w4::DeviceInfo info{};                 // constant once ready (inject is kept apart)
    unsigned int *status = nullptr;
    std::atomic<unsigned int> inject{0};  // this device's injection flags
};
DevCache g_dev[64];
std::mutex g_dev_mu;

// Current device's info and status-word address (looked up once per device).
int device_state(w4::DeviceInfo &info, unsigned int *&status, DevCache **cache = nullptr) {
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (d < 0 || d >= 64) return fail(W4A16_ERR_UNSUPPORTED, "device ordinal %d >= 64", d);
    DevCache &c = g_dev[d];
    if (!c.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!c.ready.load(std::memory_order_relaxed)) {
            w4::DeviceInfo inf{};
            inf.device = d;
            e = cudaDeviceGetAttribute(&inf.num_sms, cudaDevAttrMultiProcessorCount, d);
            if (e == cudaSuccess)
                e = cudaDeviceGetAttribute(&inf.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
            void *p = nullptr;
            if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, g_status);
            if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
            c.info = inf;
            c.status = static_cast<unsigned int *>(p);
            c.ready.store(true, std::memory_order_release);
        }
    }
    info = c.info;
    info.inject = c.inject.load(std::memory_order_relaxed);
    status = c.status;
    if (cache) *cache = &c;
    return W4A16_OK;
}

// Every data pointer must be memory of the current device (the launches go
// to the current device): device memory of that device, or managed memory.
// Null entries (an absent optional tensor) are skipped.
int check_device_ptrs(const char *who, int device, std::initializer_list<const void *> ptrs) {
    int i = 0;
    for (const void *p : ptrs) {
        ++i;
        if (!p) continue;
        cudaPointerAttributes at;
        const cudaError_t e = cudaPointerGetAttributes(&at, p);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(W4A16_ERR_INVALID_ARG, "%s: pointer %d is not CUDA memory (%s)", who, i,
                        cudaGetErrorString(e));
        }
        if (at.type == cudaMemoryTypeManaged) continue;
        if (at.type != cudaMemoryTypeDevice)
            return fail(W4A16_ERR_INVALID_ARG, "%s: pointer %d is not device memory", who, i);
        if (at.device != device)
            return fail(W4A16_ERR_INVALID_ARG, "%s: pointer %d is memory of device %d, the current device is %d", who,
                        i, at.device, device);
    }
    return W4A16_OK;
}

int launched(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
    return ok();
}

// Host checks of one INT4 linear, M = 1 (the GEMV's rules) or any M (the
// GEMM's rules); `who` prefixes the message.
int check_gemv_args(const char *who, const void *x, const void *qw, const void *s, const void *z, const void *y,
                    int64_t N, int64_t K, int group) {
    if (!x || !qw || !s || !y) return fail(W4A16_ERR_INVALID_ARG, "%s: null pointer", who);
    if (N < 1 || K < 1)
        return fail(W4A16_ERR_INVALID_ARG, "%s: N=%lld K=%lld must be >= 1", who, (long long)N, (long long)K);
    if (group != 128) return fail(W4A16_ERR_UNSUPPORTED, "%s: group %d (only 128)", who, group);
    if (K % 128 != 0) return fail(W4A16_ERR_INVALID_ARG, "%s: K=%lld not a multiple of the group", who, (long long)K);
    if (K > 16384) return fail(W4A16_ERR_UNSUPPORTED, "%s: K=%lld > 16384", who, (long long)K);
    if (N > (int64_t(1) << 31)) return fail(W4A16_ERR_UNSUPPORTED, "%s: N=%lld too large", who, (long long)N);
    if (!aligned16(x) || !aligned16(qw) || !aligned16(s) || (z && !aligned16(z)) || !aligned16(y))
        return fail(W4A16_ERR_MISALIGNED, "%s: pointers must be 16-byte aligned", who);
    return W4A16_OK;
}

int check_gemm_args(const char *who, const void *X, const void *qw, const void *s, const void *z, const void *Y,
                    int64_t M, int64_t N, int64_t K, int group) {
    if (!X || !qw || !s || !Y) return fail(W4A16_ERR_INVALID_ARG, "%s: null pointer", who);
    if (M < 1 || N < 1 || K < 1)
        return fail(W4A16_ERR_INVALID_ARG, "%s: M=%lld N=%lld K=%lld must be >= 1", who, (long long)M,
                    (long long)N, (long long)K);
    if (group != 128) return fail(W4A16_ERR_UNSUPPORTED, "%s: group %d (only 128)", who, group);
    if (K % 128 != 0) return fail(W4A16_ERR_INVALID_ARG, "%s: K=%lld not a multiple of the group", who, (long long)K);
    if (K > 16384) return fail(W4A16_ERR_UNSUPPORTED, "%s: K=%lld > 16384", who, (long long)K);
    if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || M * N > (int64_t(1) << 40))
        return fail(W4A16_ERR_UNSUPPORTED, "%s: sizes too large", who);
    if (!aligned16(X) || !aligned16(qw) || !aligned16(s) || (z && !aligned16(z)) || !aligned16(Y))
        return fail(W4A16_ERR_MISALIGNED, "%s: pointers must be 16-byte aligned", who);
    return W4A16_OK;
}

// Decode-sized batches stream the weights on the CUDA cores: M = 1 the GEMV,
// up to four rows sharing one pass (two passes where K leaves fewer teams
// per CTA).  Larger M goes to the tensor cores, whose GEMM (X tiles of M
// rounded up to 16 rows) has a fixed pipeline latency that dominates at
// small M (N = 15360, K = 3840, GEMM against streaming passes of up to four
// rows: M = 4 -- / 19.1 us, M = 5 25.0 / 26.2 us, M = 6 25.1 / 30.0 us,
// M = 8 25.0 / 36.9 us).
cudaError_t launch_int4_linear(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const uint16_t *z,
                               uint16_t *Y, int64_t M, int64_t N, int64_t K, cudaStream_t st, unsigned int *status,
                               const w4::DeviceInfo &dev) {
    if (M > 4) return w4::launch_gemm_int4(X, qw, s, z, Y, M, N, K, st, status, dev);
    const int64_t mv_max = w4::gemv_int4_max_mv(K) >= 4 ? 4 : 2;
    while (M > 0) {
        const int64_t mv = M >= mv_max ? mv_max : M >= 2 ? 2 : 1;
        const cudaError_t e = mv == 1 ? w4::launch_gemv_int4(X, qw, s, z, Y, N, K, st, status, dev)
                                      : w4::launch_gemv_int4_batched(X, qw, s, z, Y, mv, N, K, st, status, dev);
        if (e != cudaSuccess) return e;
        // the next rows (Y + mv N need not be 16-byte aligned: the GEMV
        // writes its outputs one by one)
        X += mv * K;
        Y += mv * N;
        M -= mv;
    }
    return cudaSuccess;
}

// The checks of op i of a sequence (M = 1: the GEMV's rules).
int check_linear(const w4a16_linear &op, int i, int group, const char *fn) {
    char who[96];
    snprintf(who, sizeof who, "%s: op %d", fn, i);
    if (op.M == 1) return check_gemv_args(who, op.x, op.qw, op.s, op.z, op.y, op.N, op.K, group);
    return check_gemm_args(who, op.x, op.qw, op.s, op.z, op.y, op.M, op.N, op.K, group);
}

int check_sequence(const w4a16_linear *ops, int count, int group, const char *fn) {
    if (count < 0) return fail(W4A16_ERR_INVALID_ARG, "%s: count %d < 0", fn, count);
    if (count > 0 && !ops) return fail(W4A16_ERR_INVALID_ARG, "%s: null ops", fn);
    for (int i = 0; i < count; ++i)
        if (int r = check_linear(ops[i], i, group, fn)) return r;
    return W4A16_OK;
}

int check_sequence_ptrs(const w4a16_linear *ops, int count, int device, const char *fn) {
    char who[96];
    for (int i = 0; i < count; ++i) {
        snprintf(who, sizeof who, "%s: op %d", fn, i);
        const w4a16_linear &o = ops[i];
        if (int r = check_device_ptrs(who, device, {o.x, o.qw, o.s, o.z, o.y})) return r;
    }
    return W4A16_OK;
}

// Launches every op in order; on a launch error returns it and the index.
cudaError_t launch_sequence(const w4a16_linear *ops, int count, cudaStream_t st, unsigned int *status,
                            const w4::DeviceInfo &dev, int &failed_at) {
    for (int i = 0; i < count; ++i) {
        const w4a16_linear &o = ops[i];
        cudaError_t e = launch_int4_linear(o.x, o.qw, o.s, o.z, o.y, o.M, o.N, o.K, st, status, dev);
        if (e != cudaSuccess) {
            failed_at = i;
            return e;
        }
    }
    failed_at = -1;
    return cudaSuccess;
}

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range range_of(const void *p, int64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, p ? a + static_cast<uintptr_t>(bytes) : a};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Checks a chain of M = 1 linears and fills the kernel's op table: for each
// op the last earlier op it conflicts with (it reads what that op writes,
// or writes what that op reads or writes), -1 for none.  Refused: an op
// whose output overlaps its own input, outputs that overlap any op's
// weights (weights are streamed ahead of the ops' order) or the scratch.
int plan_chain(const w4a16_linear *ops, int count, Range scratch, w4::ChainOp *plan) {
    for (int i = 0; i < count; ++i) {
        const w4a16_linear &o = ops[i];
        if (o.M != 1)
            return fail(W4A16_ERR_UNSUPPORTED, "w4a16_linear_chain: op %d has M=%lld (a chain takes M = 1 ops)", i,
                        (long long)o.M);
        if (o.N > 0x7FFFFFFF)
            return fail(W4A16_ERR_UNSUPPORTED, "w4a16_linear_chain: op %d N=%lld too large", i, (long long)o.N);
        const Range xi = range_of(o.x, 2 * o.K), yi = range_of(o.y, 2 * o.N);
        if (overlap(xi, yi)) return fail(W4A16_ERR_INVALID_ARG, "w4a16_linear_chain: op %d writes its own input", i);
        if (overlap(yi, scratch)) return fail(W4A16_ERR_INVALID_ARG, "w4a16_linear_chain: op %d writes the scratch", i);
        for (int j = 0; j < count; ++j) {
            const w4a16_linear &w = ops[j];
            const int64_t Gj = w.K / 128;
            if (overlap(yi, range_of(w.qw, w.N * w.K / 2)) || overlap(yi, range_of(w.s, 2 * w.N * Gj)) ||
                (w.z && overlap(yi, range_of(w.z, 2 * w.N * Gj))))
                return fail(W4A16_ERR_INVALID_ARG, "w4a16_linear_chain: op %d writes the weights of op %d", i, j);
        }
        w4::ChainOp &c = plan[i];
        c.x = o.x;
        c.qw = o.qw;
        c.s = o.s;
        c.z = o.z;
        c.y = o.y;
        c.N = static_cast<int>(o.N);
        c.K = static_cast<int>(o.K);
        w4::gemv_chain_shape(o.K, c.tt_log2, c.rpt);
        c.dep = -1;
        for (int j = i - 1; j >= 0; --j) {
            const Range xj = range_of(ops[j].x, 2 * ops[j].K), yj = range_of(ops[j].y, 2 * ops[j].N);
            if (overlap(yj, xi) || overlap(xj, yi) || overlap(yj, yi)) {
                c.dep = j;
                break;
            }
        }
    }
    return W4A16_OK;
}

int64_t chain_scratch_bytes(int count) {
    if (count < 1) return 0;
    const int64_t launches = (count + w4::kChainMaxOps - 1) / w4::kChainMaxOps;
    return 4 * (static_cast<int64_t>(count) + launches);
}

// Built-in scratch of w4a16_linear_chain_noalloc, for callers that cannot
// allocate device memory: 16 KB (4096 words) of completion counters; a chain
// of n linears needs n + ceil(n / 192) of them, so at most kNoAllocMaxOps.
// It exists once per device that loads this library, for as long as the
// library stays loaded.  In host code its name is not a device address: the
// address comes from cudaGetSymbolAddress, looked up once per device.
constexpr int kNoAllocMaxOps = 4032;
constexpr int kNoAllocWords = 4096;
static_assert(kNoAllocMaxOps + (kNoAllocMaxOps + w4::kChainMaxOps - 1) / w4::kChainMaxOps <= kNoAllocWords,
              "built-in scratch too small");
static __device__ __align__(256) unsigned int g_chain_noalloc_scratch[kNoAllocWords];

struct NoAllocScratch {
    std::atomic<bool> ready{false};
    unsigned int *ptr = nullptr;
};
NoAllocScratch g_noalloc[64];
std::mutex g_noalloc_mu;

// The built-in scratch's device address on `device` (the current device).
int noalloc_scratch(int device, unsigned int *&ptr) {
    NoAllocScratch &c = g_noalloc[device & 63];
    if (!c.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!c.ready.load(std::memory_order_relaxed)) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_chain_noalloc_scratch);
            if (e != cudaSuccess)
                return fail(W4A16_ERR_CUDA, "w4a16_linear_chain_noalloc: scratch address: %s", cudaGetErrorString(e));
            c.ptr = static_cast<unsigned int *>(p);
            c.ready.store(true, std::memory_order_release);
        }
    }
    ptr = c.ptr;
    return W4A16_OK;
}

// plan_chain for the ops c0 .. c0 + n - 1 of a chain of `count` (the piece
// one launch takes), with no scratch of the caller's to protect: the
// dependencies are sought within the piece (an earlier piece is finished by
// the stream order) and the indices are the piece's own.
int plan_chain_piece(const w4a16_linear *ops, int count, int c0, int n, w4::ChainOp *plan) {
    for (int i = 0; i < n; ++i) {
        const int oi = c0 + i;
        const w4a16_linear &o = ops[oi];
        if (o.M != 1)
            return fail(W4A16_ERR_UNSUPPORTED, "w4a16_linear_chain_noalloc: op %d has M=%lld (M = 1 ops only)", oi,
                        (long long)o.M);
        if (o.N > 0x7FFFFFFF)
            return fail(W4A16_ERR_UNSUPPORTED, "w4a16_linear_chain_noalloc: op %d N=%lld too large", oi,
                        (long long)o.N);
        const Range xi = range_of(o.x, 2 * o.K), yi = range_of(o.y, 2 * o.N);
        if (overlap(xi, yi))
            return fail(W4A16_ERR_INVALID_ARG, "w4a16_linear_chain_noalloc: op %d writes its own input", oi);
        for (int j = 0; j < count; ++j) {
            const w4a16_linear &w = ops[j];
            const int64_t Gj = w.K / 128;
            if (overlap(yi, range_of(w.qw, w.N * w.K / 2)) || overlap(yi, range_of(w.s, 2 * w.N * Gj)) ||
                (w.z && overlap(yi, range_of(w.z, 2 * w.N * Gj))))
                return fail(W4A16_ERR_INVALID_ARG, "w4a16_linear_chain_noalloc: op %d writes the weights of op %d", oi,
                            j);
        }
        w4::ChainOp &c = plan[i];
        c.x = o.x;
        c.qw = o.qw;
        c.s = o.s;
        c.z = o.z;
        c.y = o.y;
        c.N = static_cast<int>(o.N);
        c.K = static_cast<int>(o.K);
        w4::gemv_chain_shape(o.K, c.tt_log2, c.rpt);
        c.dep = -1;
        c.report = 0;
        c.pad = 0;
        for (int j = i - 1; j >= 0; --j) {
            const w4a16_linear &p = ops[c0 + j];
            const Range xj = range_of(p.x, 2 * p.K), yj = range_of(p.y, 2 * p.N);
            if (overlap(yj, xi) || overlap(xj, yi) || overlap(yj, yi)) {
                c.dep = j;
                break;
            }
        }
    }
    for (int i = 0; i < n; ++i)
        if (plan[i].dep >= 0) plan[plan[i].dep].report = 1;
    return W4A16_OK;
}

// Launches a planned chain in pieces of at most kChainMaxOps ops, each with
// its own counters in the scratch; a dependency on an op of an earlier piece
// is met by the stream order.
cudaError_t launch_chain(w4::ChainOp *plan, int count, unsigned int *scratch, cudaStream_t st, unsigned int *status,
                         const w4::DeviceInfo &dev) {
    unsigned int *done = scratch;
    for (int c0 = 0; c0 < count; c0 += w4::kChainMaxOps) {
        const int n = count - c0 < w4::kChainMaxOps ? count - c0 : w4::kChainMaxOps;
        w4::ChainOp *piece = plan + c0;
        for (int i = 0; i < n; ++i) {
            piece[i].dep = piece[i].dep >= c0 ? piece[i].dep - c0 : -1;
            piece[i].report = 0;
        }
        for (int i = 0; i < n; ++i)
            if (piece[i].dep >= 0) piece[piece[i].dep].report = 1;
        const cudaError_t e = w4::launch_gemv_chain(piece, n, done, st, status, dev);
        if (e != cudaSuccess) return e;
        done += n + 1;
    }
    return cudaSuccess;
}

// The address through which the current device reaches p: p itself for
// memory of this device (or managed memory), the mapped device address for
// pinned host memory; nullptr (with the message set) for anything else.
void *device_address(const char *who, const char *name, const void *p, int device) {
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        fail(W4A16_ERR_INVALID_ARG, "%s: %s is not CUDA memory (%s)", who, name, cudaGetErrorString(e));
        return nullptr;
    }
    if (at.type == cudaMemoryTypeManaged) return const_cast<void *>(p);
    if (at.type == cudaMemoryTypeDevice) {
        if (at.device != device) {
            fail(W4A16_ERR_INVALID_ARG, "%s: %s is memory of device %d, the current device is %d", who, name,
                 at.device, device);
            return nullptr;
        }
        return const_cast<void *>(p);
    }
    if (at.type == cudaMemoryTypeHost && at.devicePointer) return at.devicePointer;
    fail(W4A16_ERR_INVALID_ARG, "%s: %s is host memory the device cannot reach (pageable, or pinned unmapped)", who,
         name);
    return nullptr;
}

}  // namespace

extern "C" {

int w4a16_version(void) { return 1 * 10000 + 1 * 100 + 0; }

const char *w4a16_last_error_string(void) { return g_err; }

int w4a16_gemv(const uint16_t *x, const uint8_t *qw, const uint16_t *s,
               const uint16_t *z, uint16_t *y, int64_t N, int64_t K,
               int group, void *stream) {
    if (int r = check_gemv_args("w4a16_gemv", x, qw, s, z, y, N, K, group)) return r;
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_device_ptrs("w4a16_gemv", dev.device, {x, qw, s, z, y})) return r;
    return launched(w4::launch_gemv_int4(x, qw, s, z, y, N, K, static_cast<cudaStream_t>(stream), status, dev),
                    "w4a16_gemv");
}

int w4a16_gemm(const uint16_t *X, const uint8_t *qw, const uint16_t *s,
               const uint16_t *z, uint16_t *Y, int64_t M, int64_t N,
               int64_t K, int group, void *stream) {
    if (int r = check_gemm_args("w4a16_gemm", X, qw, s, z, Y, M, N, K, group)) return r;
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_device_ptrs("w4a16_gemm", dev.device, {X, qw, s, z, Y})) return r;
    return launched(launch_int4_linear(X, qw, s, z, Y, M, N, K, static_cast<cudaStream_t>(stream), status, dev),
                    "w4a16_gemm");
}

int w4a16_gemm_f16(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const uint16_t *z, uint16_t *Y,
                   int64_t M, int64_t N, int64_t K, int group, void *stream) {
    const char *fn = "w4a16_gemm_f16";
    if (int r = check_gemm_args(fn, X, qw, s, z, Y, M, N, K, group)) return r;
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_device_ptrs(fn, dev.device, {X, qw, s, z, Y})) return r;
    return launched(w4::launch_gemm_int4_f16(X, qw, s, z, Y, M, N, K, static_cast<cudaStream_t>(stream), status, dev),
                    fn);
}

int w4a16_copy(void *dst, const void *src, int64_t bytes, void *stream) {
    const char *fn = "w4a16_copy";
    if (bytes < 0) return fail(W4A16_ERR_INVALID_ARG, "%s: bytes=%lld < 0", fn, (long long)bytes);
    if (bytes == 0) return ok();  // nothing to copy (an empty buffer's pointer may be null)
    if (!dst || !src) return fail(W4A16_ERR_INVALID_ARG, "%s: null pointer", fn);
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    void *d = device_address(fn, "dst", dst, dev.device);
    if (!d) return W4A16_ERR_INVALID_ARG;
    void *sp = device_address(fn, "src", src, dev.device);
    if (!sp) return W4A16_ERR_INVALID_ARG;
    return launched(w4::launch_copy(d, sp, bytes, static_cast<cudaStream_t>(stream), dev), fn);
}

int w4a16_bf16_gemm(const uint16_t *X, const uint16_t *W, uint16_t *Y, int64_t M, int64_t N, int64_t K,
                    void *stream) {
    if (!X || !W || !Y) return fail(W4A16_ERR_INVALID_ARG, "w4a16_bf16_gemm: null pointer");
    if (M < 1 || N < 1 || K < 1)
        return fail(W4A16_ERR_INVALID_ARG, "w4a16_bf16_gemm: M=%lld N=%lld K=%lld must be >= 1", (long long)M,
                    (long long)N, (long long)K);
    if (K % 64 != 0) return fail(W4A16_ERR_INVALID_ARG, "w4a16_bf16_gemm: K=%lld not a multiple of 64", (long long)K);
    if (K > (int64_t(1) << 20) || M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || M * N > (int64_t(1) << 40))
        return fail(W4A16_ERR_UNSUPPORTED, "w4a16_bf16_gemm: sizes too large");
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y))
        return fail(W4A16_ERR_MISALIGNED, "w4a16_bf16_gemm: pointers must be 16-byte aligned");
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_device_ptrs("w4a16_bf16_gemm", dev.device, {X, W, Y})) return r;
    return launched(w4::launch_bf16_gemm(X, W, Y, M, N, K, static_cast<cudaStream_t>(stream), status, dev),
                    "w4a16_bf16_gemm");
}

int fp4_moe_gemv(const uint16_t *x, const uint8_t *qw, const uint16_t *s,
                 const int32_t *expert_ids, int topk, uint16_t *y, int64_t E,
                 int64_t N, int64_t K, int group, void *stream) {
    if (!x || !qw || !s || !expert_ids || !y) return fail(W4A16_ERR_INVALID_ARG, "fp4_moe_gemv: null pointer");
    if (topk < 1 || E < 1 || N < 1 || K < 1)
        return fail(W4A16_ERR_INVALID_ARG, "fp4_moe_gemv: topk=%d E=%lld N=%lld K=%lld must be >= 1", topk,
                    (long long)E, (long long)N, (long long)K);
    if (group != 32) return fail(W4A16_ERR_UNSUPPORTED, "fp4_moe_gemv: group %d (only 32)", group);
    if (K % 64 != 0) return fail(W4A16_ERR_INVALID_ARG, "fp4_moe_gemv: K=%lld not a multiple of 64", (long long)K);
    if (K > 16384) return fail(W4A16_ERR_UNSUPPORTED, "fp4_moe_gemv: K=%lld > 16384", (long long)K);
    if (E * N > (int64_t(1) << 31) || (int64_t)topk * N > (int64_t(1) << 31))
        return fail(W4A16_ERR_UNSUPPORTED, "fp4_moe_gemv: sizes too large");
    if (!aligned16(x) || !aligned16(qw) || !aligned16(s) || !aligned16(y))
        return fail(W4A16_ERR_MISALIGNED, "fp4_moe_gemv: pointers must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(expert_ids) & 3u) != 0)
        return fail(W4A16_ERR_MISALIGNED, "fp4_moe_gemv: expert_ids must be 4-byte aligned");
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_device_ptrs("fp4_moe_gemv", dev.device, {x, qw, s, expert_ids, y})) return r;
    return launched(w4::launch_moe_fp4(x, qw, s, expert_ids, topk, y, E, N, K, static_cast<cudaStream_t>(stream),
                                       status, dev),
                    "fp4_moe_gemv");
}

int64_t fp4_moe_gemm_scratch_bytes(int M, int topk, int64_t E, int64_t K) {
    if (M < 1 || topk < 1 || E < 1 || K < 1) return 0;
    return w4::moe_fp4_gemm_scratch(static_cast<int64_t>(M) * topk, E, K);
}

int fp4_moe_gemm(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const int32_t *expert_ids, int M,
                 int topk, uint16_t *Y, int64_t E, int64_t N, int64_t K, int group, void *scratch,
                 int64_t scratch_bytes, void *stream) {
    const char *fn = "fp4_moe_gemm";
    if (!X || !qw || !s || !expert_ids || !Y || !scratch) return fail(W4A16_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (M < 1 || topk < 1 || E < 1 || N < 1 || K < 1)
        return fail(W4A16_ERR_INVALID_ARG, "%s: M=%d topk=%d E=%lld N=%lld K=%lld must be >= 1", fn, M, topk,
                    (long long)E, (long long)N, (long long)K);
    if (group != 32) return fail(W4A16_ERR_UNSUPPORTED, "%s: group %d (only 32)", fn, group);
    if (K % 256 != 0) return fail(W4A16_ERR_UNSUPPORTED, "%s: K=%lld not a multiple of 256", fn, (long long)K);
    if (K > 65536 || E > 8192 || E * N > (int64_t(1) << 31) - 128 || static_cast<int64_t>(M) * topk > (1 << 20))
        return fail(W4A16_ERR_UNSUPPORTED, "%s: sizes too large", fn);
    if (!aligned16(X) || !aligned16(qw) || !aligned16(s) || !aligned16(Y))
        return fail(W4A16_ERR_MISALIGNED, "%s: pointers must be 16-byte aligned", fn);
    if ((reinterpret_cast<uintptr_t>(expert_ids) & 3u) != 0)
        return fail(W4A16_ERR_MISALIGNED, "%s: expert_ids must be 4-byte aligned", fn);
    if ((reinterpret_cast<uintptr_t>(scratch) & 255u) != 0)
        return fail(W4A16_ERR_MISALIGNED, "%s: scratch must be 256-byte aligned", fn);
    const int64_t need = w4::moe_fp4_gemm_scratch(static_cast<int64_t>(M) * topk, E, K);
    if (scratch_bytes < need)
        return fail(W4A16_ERR_INVALID_ARG, "%s: scratch of %lld bytes, %lld needed", fn, (long long)scratch_bytes,
                    (long long)need);
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_device_ptrs(fn, dev.device, {X, qw, s, expert_ids, Y, scratch})) return r;
    return launched(w4::launch_moe_fp4_gemm(X, qw, s, expert_ids, M, topk, Y, E, N, K, scratch,
                                            static_cast<cudaStream_t>(stream), status, dev),
                    fn);
}

int w4a16_dequant(int fmt, const uint8_t *qw, const uint16_t *s,
                  const uint16_t *z, void *out, int out_dtype, int64_t rows,
                  int64_t K, int group, void *stream) {
    if (fmt != W4_FMT_INT4_ASYM && fmt != W4_FMT_FP4_E2M1)
        return fail(W4A16_ERR_INVALID_ARG, "w4a16_dequant: unknown format %d", fmt);
    if (out_dtype != W4_OUT_F32 && out_dtype != W4_OUT_BF16)
        return fail(W4A16_ERR_INVALID_ARG, "w4a16_dequant: unknown output dtype %d", out_dtype);
    if (!qw || !s || !out) return fail(W4A16_ERR_INVALID_ARG, "w4a16_dequant: null pointer");
    if (fmt == W4_FMT_FP4_E2M1 && z) return fail(W4A16_ERR_INVALID_ARG, "w4a16_dequant: FP4 takes no z");
    if (rows < 1 || K < 1) return fail(W4A16_ERR_INVALID_ARG, "w4a16_dequant: rows, K must be >= 1");
    const int want = fmt == W4_FMT_INT4_ASYM ? 128 : 32;
    if (group != want) return fail(W4A16_ERR_UNSUPPORTED, "w4a16_dequant: group %d (need %d)", group, want);
    if (K % group != 0) return fail(W4A16_ERR_INVALID_ARG, "w4a16_dequant: K %% group != 0");
    if (!aligned16(qw) || !aligned16(s) || (z && !aligned16(z)) || !aligned16(out))
        return fail(W4A16_ERR_MISALIGNED, "w4a16_dequant: pointers must be 16-byte aligned");
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_device_ptrs("w4a16_dequant", dev.device, {qw, s, z, out})) return r;
    (void)status;
    return launched(w4::launch_dequant(fmt, qw, s, z, out, out_dtype, rows, K, group,
                                       static_cast<cudaStream_t>(stream), dev),
                    "w4a16_dequant");
}

int64_t w4a16_linear_chain_scratch_bytes(int count) { return chain_scratch_bytes(count); }

int w4a16_linear_chain(const w4a16_linear *ops, int count, int group, void *scratch, int64_t scratch_bytes,
                       void *stream) {
    if (int r = check_sequence(ops, count, group, "w4a16_linear_chain")) return r;
    if (count == 0) return ok();
    if (!scratch) return fail(W4A16_ERR_INVALID_ARG, "w4a16_linear_chain: null scratch");
    if ((reinterpret_cast<uintptr_t>(scratch) & 3u) != 0)
        return fail(W4A16_ERR_MISALIGNED, "w4a16_linear_chain: scratch must be 4-byte aligned");
    const int64_t need = chain_scratch_bytes(count);
    if (scratch_bytes < need)
        return fail(W4A16_ERR_INVALID_ARG, "w4a16_linear_chain: scratch of %lld bytes, %lld needed",
                    (long long)scratch_bytes, (long long)need);
    w4::ChainOp *plan = new (std::nothrow) w4::ChainOp[count];
    if (!plan) return fail(W4A16_ERR_CUDA, "w4a16_linear_chain: out of host memory");
    int r = plan_chain(ops, count, range_of(scratch, need), plan);
    w4::DeviceInfo dev;
    unsigned int *status = nullptr;
    if (!r) r = device_state(dev, status);
    if (!r) r = check_sequence_ptrs(ops, count, dev.device, "w4a16_linear_chain");
    if (!r) r = check_device_ptrs("w4a16_linear_chain: scratch", dev.device, {scratch});
    if (!r) {
        const cudaError_t e = launch_chain(plan, count, static_cast<unsigned int *>(scratch),
                                           static_cast<cudaStream_t>(stream), status, dev);
        r = launched(e, "w4a16_linear_chain");
    }
    delete[] plan;
    return r;
}

int w4a16_linear_chain_noalloc(const w4a16_linear *ops, int count, int group, void *stream) {
    if (int r = check_sequence(ops, count, group, "w4a16_linear_chain_noalloc")) return r;
    if (count == 0) return ok();
    if (count > kNoAllocMaxOps)
        return fail(W4A16_ERR_UNSUPPORTED,
                    "w4a16_linear_chain_noalloc: %d linears; its built-in scratch holds the counters of at most %d "
                    "(use w4a16_linear_chain with scratch of your own)",
                    count, kNoAllocMaxOps);
    w4::DeviceInfo dev;
    unsigned int *status = nullptr;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_sequence_ptrs(ops, count, dev.device, "w4a16_linear_chain_noalloc")) return r;
    unsigned int *scratch = nullptr;
    if (int r = noalloc_scratch(dev.device, scratch)) return r;
    // every op checked (and its dependencies found) before anything is queued
    w4::ChainOp piece[w4::kChainMaxOps];
    for (int c0 = 0; c0 < count; c0 += w4::kChainMaxOps) {
        const int n = count - c0 < w4::kChainMaxOps ? count - c0 : w4::kChainMaxOps;
        if (int r = plan_chain_piece(ops, count, c0, n, piece)) return r;
    }
    // the counters must start at zero; the array keeps whatever the last call
    // left, so clear them in stream order before the launches
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(scratch, 0, static_cast<size_t>(chain_scratch_bytes(count)), st);
    if (e != cudaSuccess)
        return fail(W4A16_ERR_CUDA, "w4a16_linear_chain_noalloc: clearing the counters: %s", cudaGetErrorString(e));
    unsigned int *done = scratch;
    for (int c0 = 0; c0 < count; c0 += w4::kChainMaxOps) {
        const int n = count - c0 < w4::kChainMaxOps ? count - c0 : w4::kChainMaxOps;
        plan_chain_piece(ops, count, c0, n, piece);  // checked above
        e = w4::launch_gemv_chain(piece, n, done, st, status, dev);
        if (e != cudaSuccess) return launched(e, "w4a16_linear_chain_noalloc");
        done += n + 1;
    }
    return ok();
}

int w4a16_linear_sequence(const w4a16_linear *ops, int count, int group, void *stream) {
    if (int r = check_sequence(ops, count, group, "w4a16_linear_sequence")) return r;
    if (count == 0) return ok();
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_sequence_ptrs(ops, count, dev.device, "w4a16_linear_sequence")) return r;
    int at = -1;
    cudaError_t e = launch_sequence(ops, count, static_cast<cudaStream_t>(stream), status, dev, at);
    if (e != cudaSuccess)
        return fail(W4A16_ERR_CUDA, "w4a16_linear_sequence: op %d launch: %s (ops before it queued)", at,
                    cudaGetErrorString(e));
    return ok();
}

}  // extern "C"

struct w4a16_graph_s {
    cudaGraphExec_t exec;
    int device;
};

extern "C" {

int w4a16_graph_create(const w4a16_linear *ops, int count, int group, w4a16_graph_t *out) {
    if (!out) return fail(W4A16_ERR_INVALID_ARG, "w4a16_graph_create: null handle pointer");
    *out = nullptr;
    if (count < 1) return fail(W4A16_ERR_INVALID_ARG, "w4a16_graph_create: count %d < 1", count);
    if (int r = check_sequence(ops, count, group, "w4a16_graph_create")) return r;
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    if (int r = check_sequence_ptrs(ops, count, dev.device, "w4a16_graph_create")) return r;
    cudaStream_t cs = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "w4a16_graph_create: stream: %s", cudaGetErrorString(e));
    // relaxed capture: a launcher's first call per kernel sets the kernel's
    // shared-memory attribute, which is not a stream operation
    e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
    if (e != cudaSuccess) {
        cudaStreamDestroy(cs);
        return fail(W4A16_ERR_CUDA, "w4a16_graph_create: begin capture: %s", cudaGetErrorString(e));
    }
    int at = -1;
    const cudaError_t le = launch_sequence(ops, count, cs, status, dev, at);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (le != cudaSuccess || e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();  // the launch error is reported here, not left pending
        if (le != cudaSuccess)
            return fail(W4A16_ERR_CUDA, "w4a16_graph_create: op %d launch: %s", at, cudaGetErrorString(le));
        return fail(W4A16_ERR_CUDA, "w4a16_graph_create: end capture: %s", cudaGetErrorString(e));
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "w4a16_graph_create: instantiate: %s", cudaGetErrorString(e));
    w4a16_graph_s *h = new (std::nothrow) w4a16_graph_s;
    if (!h) {
        cudaGraphExecDestroy(exec);
        return fail(W4A16_ERR_CUDA, "w4a16_graph_create: out of host memory");
    }
    h->exec = exec;
    h->device = dev.device;
    *out = h;
    return ok();
}

int w4a16_graph_launch(w4a16_graph_t graph, void *stream) {
    if (!graph) return fail(W4A16_ERR_INVALID_ARG, "w4a16_graph_launch: null graph");
    const cudaError_t e = cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(W4A16_ERR_CUDA, "w4a16_graph_launch (graph of device %d): %s", graph->device,
                    cudaGetErrorString(e));
    return ok();
}

int w4a16_graph_destroy(w4a16_graph_t graph) {
    if (!graph) return ok();
    // an executable graph still running is released when it completes
    const cudaError_t e = cudaGraphExecDestroy(graph->exec);
    delete graph;
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "w4a16_graph_destroy: %s", cudaGetErrorString(e));
    return ok();
}

int w4a16_check_device_error(void *stream) {
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_status, &zero, sizeof zero);
        if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    }
    if (v & w4::kDevTimeout) return fail(W4A16_ERR_TIMEOUT, "a device pipeline wait timed out");
    if (v & w4::kDevBadExpert) return fail(W4A16_ERR_DEVICE, "an expert id was outside [0, E)");
    return ok();
}

int w4a16_debug_inject(unsigned int flags) {
    w4::DeviceInfo dev;
    unsigned int *status;
    DevCache *c = nullptr;
    if (int r = device_state(dev, status, &c)) return r;
    if (flags & ~static_cast<unsigned int>(w4::kInjectStallPipeline | w4::kInjectStallConsumers))
        return fail(W4A16_ERR_INVALID_ARG, "unknown injection flags 0x%x", flags);
    // the flags travel as a kernel argument of later launches: the normal
    // path reads no memory for them
    c->inject.store(flags, std::memory_order_relaxed);
    return ok();
}

}  // extern "C"
