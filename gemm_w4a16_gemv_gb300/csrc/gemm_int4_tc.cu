// Prefill GEMM (M >= 1) with INT4 group-128 weights on the tcgen05 tensor
// cores.  (Kernel body added separately.)
#include "common.cuh"
#include "kernels.h"

namespace w4 {

cudaError_t launch_gemm_int4(const uint16_t *, const uint8_t *, const uint16_t *, const uint16_t *, uint16_t *,
                             int64_t, int64_t, int64_t, cudaStream_t, unsigned int *, const DeviceInfo &) {
    return cudaErrorNotSupported;
}

}  // namespace w4
