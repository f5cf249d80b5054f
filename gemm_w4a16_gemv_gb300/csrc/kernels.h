// Internal launchers, one per kernel family.  Arguments are validated by the
// C-ABI layer (api.cu) before these are called.
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

namespace w4 {

// A kernel's dynamic shared-memory limit, raised once per device to the
// largest size launched so far.  Host threads may launch concurrently, so the
// record is kept under a mutex.  `check` (optional) runs once per device
// before the first raise and may refuse the kernel.
struct SmemLimit {
    std::mutex mu;
    int bytes[64] = {};
    template <typename Check>
    cudaError_t ensure(const void *kern, int device, int need, Check check) {
        std::lock_guard<std::mutex> lk(mu);
        const int d = device & 63;
        if (bytes[d] >= need) return cudaSuccess;
        if (bytes[d] == 0) {
            const cudaError_t e = check();
            if (e != cudaSuccess) return e;
        }
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, need);
        if (e == cudaSuccess) bytes[d] = need;
        return e;
    }
    cudaError_t ensure(const void *kern, int device, int need) {
        return ensure(kern, device, need, [] { return cudaSuccess; });
    }
};

struct DeviceInfo {
    int device;
    int num_sms;
    int max_smem_optin;
    unsigned int inject;  // test-only injection flags (w4a16_debug_inject), normally 0
};

cudaError_t launch_dequant(int fmt, const uint8_t *qw, const uint16_t *s,
                           const uint16_t *z, void *out, int out_dtype,
                           int64_t rows, int64_t K, int group,
                           cudaStream_t st, const DeviceInfo &dev);

cudaError_t launch_gemv_int4(const uint16_t *x, const uint8_t *qw,
                             const uint16_t *s, const uint16_t *z, uint16_t *y,
                             int64_t N, int64_t K, cudaStream_t st,
                             unsigned int *status, const DeviceInfo &dev);

// Activation rows one INT4 streaming pass can share at this K (2 or more).
int gemv_int4_max_mv(int64_t K);

// M = 2..4 rows through the streaming GEMV (one pass over the weights).
cudaError_t launch_gemv_int4_batched(const uint16_t *X, const uint8_t *qw,
                                     const uint16_t *s, const uint16_t *z, uint16_t *Y,
                                     int64_t M, int64_t N, int64_t K, cudaStream_t st,
                                     unsigned int *status, const DeviceInfo &dev);

// One INT4 linear of a chain (M = 1), as the chain kernel reads it.
struct ChainOp {
    const uint16_t *x;
    const uint8_t *qw;
    const uint16_t *s;
    const uint16_t *z;  // null: symmetric INT4
    uint16_t *y;
    int N, K;
    int dep;                // op of the same launch that must be finished everywhere first (-1: none)
    unsigned char tt_log2;  // log2 of the threads per row (one thread per 128-code group)
    unsigned char rpt;      // rows per thread per stage (1 or 2)
    unsigned char report;   // a later op of the launch depends on this one: count its completion
    unsigned char pad;
};
constexpr int kChainMaxOps = 192;  // ops per launch (kernel parameter space)
// The team shape of an op with K columns: threads per row (log2) and rows
// per thread, as the single GEMV chooses them.
void gemv_chain_shape(int64_t K, unsigned char &tt_log2, unsigned char &rpt);
// A chain of count <= kChainMaxOps ops in one persistent launch; `done`:
// count + 1 zeroed counters in device memory (left zeroed).  ops[i].dep and
// ops[i].report index ops of this launch.
cudaError_t launch_gemv_chain(const ChainOp *ops, int count, unsigned int *done, cudaStream_t st,
                              unsigned int *status, const DeviceInfo &dev);

// Batched-expert FP4 GEMM (M tokens x topk experts): scratch bytes needed
// for P = M * topk pairs, and the three launches (route, gather, GEMM).
int64_t moe_fp4_gemm_scratch(int64_t P, int64_t E, int64_t K);
cudaError_t launch_moe_fp4_gemm(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const int32_t *ids, int M,
                                int topk, uint16_t *Y, int64_t E, int64_t N, int64_t K, void *scratch,
                                cudaStream_t st, unsigned int *status, const DeviceInfo &dev);

cudaError_t launch_moe_fp4(const uint16_t *x, const uint8_t *qw,
                           const uint16_t *s, const int32_t *ids, int topk,
                           uint16_t *y, int64_t E, int64_t N, int64_t K,
                           cudaStream_t st, unsigned int *status,
                           const DeviceInfo &dev);

// INT4 prefill GEMM with binary16 operands (pre-pass of X into
// stream-ordered scratch, then one accumulator over all of K).
int gemm_int4_f16_smem(int64_t M, int64_t K, bool sym);
cudaError_t launch_gemm_int4_f16(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const uint16_t *z,
                                 uint16_t *Y, int64_t M, int64_t N, int64_t K, cudaStream_t st, unsigned int *status,
                                 const DeviceInfo &dev);

cudaError_t launch_gemm_int4(const uint16_t *X, const uint8_t *qw,
                             const uint16_t *s, const uint16_t *z, uint16_t *Y,
                             int64_t M, int64_t N, int64_t K, cudaStream_t st,
                             unsigned int *status, const DeviceInfo &dev);

// Dense BF16 GEMM Y = X W^T (the second pass of the unfused path).
cudaError_t launch_bf16_gemm(const uint16_t *X, const uint16_t *W, uint16_t *Y,
                             int64_t M, int64_t N, int64_t K, cudaStream_t st,
                             unsigned int *status, const DeviceInfo &dev);

// dst[0, bytes) = src[0, bytes) by a kernel (addresses the device can
// dereference, already translated and checked by the caller).
cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, cudaStream_t st, const DeviceInfo &dev);

}  // namespace w4
