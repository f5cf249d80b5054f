// Small copies as a kernel: the step's activation in (pinned host -> device)
// and its result out (device -> pinned host) of a decode step, so that they
// join the chain of launches made with programmatic dependent launch instead
// of being copy-engine operations between them.  The pointers are addresses
// the device can dereference (device or managed memory, or pinned host
// memory through its mapped device address); the host entry translates and
// checks them before launching.
#include "common.cuh"
#include "kernels.h"

namespace w4 {
namespace {

constexpr int COPY_THREADS = 256;

// dst[0, bytes) = src[0, bytes): 16-byte moves when both ends are 16-byte
// aligned, the rest (or everything, when they are not) byte by byte.
__global__ void __launch_bounds__(COPY_THREADS) copy_kernel(unsigned char *dst, const unsigned char *src,
                                                            int64_t bytes) {
    pdl_launch_dependents();
    pdl_wait();  // the source (and the destination's previous users) follow the stream order
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
    const int64_t n16 = vec ? bytes / 16 : 0;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * COPY_THREADS + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * COPY_THREADS;
    for (int64_t i = tid; i < n16; i += nth) reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(src)[i];
    for (int64_t i = n16 * 16 + tid; i < bytes; i += nth) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, cudaStream_t st, const DeviceInfo &dev) {
    if (bytes <= 0) return cudaSuccess;
    const int64_t units = (bytes + 15) / 16;
    int64_t grid = (units + COPY_THREADS - 1) / COPY_THREADS;
    const int64_t cap = 4 * static_cast<int64_t>(dev.num_sms);
    if (grid > cap) grid = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(COPY_THREADS);
    cfg.stream = st;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_kernel, static_cast<unsigned char *>(dst),
                              static_cast<const unsigned char *>(src), bytes);
}

}  // namespace w4
