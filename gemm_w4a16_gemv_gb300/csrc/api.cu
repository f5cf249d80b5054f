// C ABI (include/w4a16.h): argument checks on the host, then one launch.
// Nothing here allocates device memory or synchronises except
// w4a16_check_device_error, which synchronises the given stream by design.
#include <cstdarg>
#include <cstdio>
#include <cstring>

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

struct DevCache {
    bool ready;
    w4::DeviceInfo info;  // info.inject: this device's injection flags
    unsigned int *status;
};
DevCache g_dev[64];

// Current device's info and status-word address (looked up once per device).
int device_state(w4::DeviceInfo &info, unsigned int *&status, DevCache **cache = nullptr) {
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (d < 0 || d >= 64) return fail(W4A16_ERR_UNSUPPORTED, "device ordinal %d >= 64", d);
    DevCache &c = g_dev[d];
    if (!c.ready) {
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
        c.ready = true;
    }
    info = c.info;
    status = c.status;
    if (cache) *cache = &c;
    return W4A16_OK;
}

int launched(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(W4A16_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
    return ok();
}

}  // namespace

extern "C" {

int w4a16_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char *w4a16_last_error_string(void) { return g_err; }

int w4a16_gemv(const uint16_t *x, const uint8_t *qw, const uint16_t *s,
               const uint16_t *z, uint16_t *y, int64_t N, int64_t K,
               int group, void *stream) {
    if (!x || !qw || !s || !y) return fail(W4A16_ERR_INVALID_ARG, "w4a16_gemv: null pointer");
    if (N < 1 || K < 1) return fail(W4A16_ERR_INVALID_ARG, "w4a16_gemv: N=%lld K=%lld must be >= 1", (long long)N, (long long)K);
    if (group != 128) return fail(W4A16_ERR_UNSUPPORTED, "w4a16_gemv: group %d (only 128)", group);
    if (K % 128 != 0) return fail(W4A16_ERR_INVALID_ARG, "w4a16_gemv: K=%lld not a multiple of the group", (long long)K);
    if (K > 16384) return fail(W4A16_ERR_UNSUPPORTED, "w4a16_gemv: K=%lld > 16384", (long long)K);
    if (N > (int64_t(1) << 31)) return fail(W4A16_ERR_UNSUPPORTED, "w4a16_gemv: N=%lld too large", (long long)N);
    if (!aligned16(x) || !aligned16(qw) || !aligned16(s) || (z && !aligned16(z)) || !aligned16(y))
        return fail(W4A16_ERR_MISALIGNED, "w4a16_gemv: pointers must be 16-byte aligned");
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    return launched(w4::launch_gemv_int4(x, qw, s, z, y, N, K, static_cast<cudaStream_t>(stream), status, dev),
                    "w4a16_gemv");
}

int w4a16_gemm(const uint16_t *X, const uint8_t *qw, const uint16_t *s,
               const uint16_t *z, uint16_t *Y, int64_t M, int64_t N,
               int64_t K, int group, void *stream) {
    if (!X || !qw || !s || !Y) return fail(W4A16_ERR_INVALID_ARG, "w4a16_gemm: null pointer");
    if (M < 1 || N < 1 || K < 1)
        return fail(W4A16_ERR_INVALID_ARG, "w4a16_gemm: M=%lld N=%lld K=%lld must be >= 1", (long long)M,
                    (long long)N, (long long)K);
    if (group != 128) return fail(W4A16_ERR_UNSUPPORTED, "w4a16_gemm: group %d (only 128)", group);
    if (K % 128 != 0) return fail(W4A16_ERR_INVALID_ARG, "w4a16_gemm: K=%lld not a multiple of the group", (long long)K);
    if (N % 16 != 0) return fail(W4A16_ERR_UNSUPPORTED, "w4a16_gemm: N=%lld not a multiple of 16", (long long)N);
    if (K > 16384) return fail(W4A16_ERR_UNSUPPORTED, "w4a16_gemm: K=%lld > 16384", (long long)K);
    if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || M * N > (int64_t(1) << 40))
        return fail(W4A16_ERR_UNSUPPORTED, "w4a16_gemm: sizes too large");
    if (!aligned16(X) || !aligned16(qw) || !aligned16(s) || (z && !aligned16(z)) || !aligned16(Y))
        return fail(W4A16_ERR_MISALIGNED, "w4a16_gemm: pointers must be 16-byte aligned");
    w4::DeviceInfo dev;
    unsigned int *status;
    if (int r = device_state(dev, status)) return r;
    // decode-sized batches stream the weights once on the CUDA cores; larger
    // M goes to the tensor cores
    if (M == 1)
        return launched(w4::launch_gemv_int4(X, qw, s, z, Y, N, K, static_cast<cudaStream_t>(stream), status, dev),
                        "w4a16_gemm (M = 1)");
    if (M <= 4)
        return launched(
            w4::launch_gemv_int4_batched(X, qw, s, z, Y, M, N, K, static_cast<cudaStream_t>(stream), status, dev),
            "w4a16_gemm (M <= 4)");
    return launched(w4::launch_gemm_int4(X, qw, s, z, Y, M, N, K, static_cast<cudaStream_t>(stream), status, dev),
                    "w4a16_gemm");
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
    return launched(w4::launch_moe_fp4(x, qw, s, expert_ids, topk, y, E, N, K, static_cast<cudaStream_t>(stream),
                                       status, dev),
                    "fp4_moe_gemv");
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
    (void)status;
    return launched(w4::launch_dequant(fmt, qw, s, z, out, out_dtype, rows, K, group,
                                       static_cast<cudaStream_t>(stream), dev),
                    "w4a16_dequant");
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
    if (flags & ~static_cast<unsigned int>(w4::kInjectStallPipeline))
        return fail(W4A16_ERR_INVALID_ARG, "unknown injection flags 0x%x", flags);
    // the flags travel as a kernel argument of later launches: the normal
    // path reads no memory for them
    c->info.inject = flags;
    return ok();
}

}  // extern "C"
