// Batched-expert FP4 GEMV for one token:
//   y[i, n] = sum_k x[k] * e2m1(q[ids[i], n, k]) * s[ids[i], n, k/32]
// ("DeepSeek V4 Triton FP4 optimisation in practice": six routed experts per
// token; stacking the expert weights on the host cost 20% end to end, so all
// experts are computed in one launch straight from the resident stack).
// Output rows are virtual rows v = i*N + n; the producer of the streaming
// pipeline (gemv_kernel.cuh) resolves expert ids on the device, and an id
// outside [0, E) gives a zero row and sets the device status.
#include "gemv_kernel.cuh"
#include "kernels.h"

namespace w4 {

cudaError_t launch_moe_fp4(const uint16_t *x, const uint8_t *qw, const uint16_t *s, const int32_t *ids,
                           int topk, uint16_t *y, int64_t E, int64_t N, int64_t K, cudaStream_t st,
                           unsigned int *status, const DeviceInfo &dev) {
    GemvParams a{};
    a.x = x;
    a.qw = qw;
    a.s = s;
    a.z = nullptr;
    a.ids = ids;
    a.y = y;
    a.status = status;
    a.inject = dev.inject;
    a.rows_per_slot = N;
    a.V = static_cast<int64_t>(topk) * N;
    a.E = E;
    a.sz_total = E * N * (K / 32) * 2;
    a.K = static_cast<int>(K);
    a.G = static_cast<int>(K / 32);
    return gemv_dispatch<true>(a, st, dev.device, dev.num_sms, dev.max_smem_optin);
}

}  // namespace w4
