// M = 1 decode GEMV with INT4 group-128 weights:
//   y[n] = sum_k x[k] * (q[n,k] - z[n,k/128]) * s[n,k/128]
// (asymmetric; symmetric INT4 passes no zero points and takes z = 8)
// ("Lab 5: Gemma4 end-to-end inference optimisation", section "INT4 fused
// GEMV": the packed weight is read once, unpacked in registers, scaled and
// zero-shifted per group and dotted with the activation, never written back).
// The streaming pipeline itself is in gemv_kernel.cuh.
#include "gemv_kernel.cuh"
#include "kernels.h"

namespace w4 {

cudaError_t launch_gemv_int4(const uint16_t *x, const uint8_t *qw, const uint16_t *s, const uint16_t *z,
                             uint16_t *y, int64_t N, int64_t K, cudaStream_t st, unsigned int *status,
                             const DeviceInfo &dev) {
    GemvParams a{};
    a.x = x;
    a.qw = qw;
    a.s = s;
    a.z = z;
    a.ids = nullptr;
    a.y = y;
    a.status = status;
    a.inject = dev.inject;
    a.rows_per_slot = N;
    a.V = N;
    a.E = 1;
    a.sz_total = N * (K / 128) * 2;
    a.K = static_cast<int>(K);
    a.G = static_cast<int>(K / 128);
    return z ? gemv_dispatch<false, false>(a, st, dev.device, dev.num_sms, dev.max_smem_optin)
             : gemv_dispatch<false, true>(a, st, dev.device, dev.num_sms, dev.max_smem_optin);
}

int gemv_int4_max_mv(int64_t K) { return gemv_int4_teams(K); }

// Batched decode: M = 2..4 activation rows X [M, K] against one pass over the
// weights (the rows share every weight stage), Y [M, N].
cudaError_t launch_gemv_int4_batched(const uint16_t *X, const uint8_t *qw, const uint16_t *s, const uint16_t *z,
                                     uint16_t *Y, int64_t M, int64_t N, int64_t K, cudaStream_t st,
                                     unsigned int *status, const DeviceInfo &dev) {
    if (M < 2 || M > 4) return cudaErrorInvalidValue;
    GemvParams a{};
    a.x = X;
    a.qw = qw;
    a.s = s;
    a.z = z;
    a.ids = nullptr;
    a.y = Y;
    a.status = status;
    a.inject = dev.inject;
    a.rows_per_slot = N;
    a.V = N;
    a.E = 1;
    a.sz_total = N * (K / 128) * 2;
    a.K = static_cast<int>(K);
    a.G = static_cast<int>(K / 128);
    a.ldy = N;
    a.mv_valid = static_cast<int>(M);
    if (M == 2)
        return z ? gemv_dispatch<false, false, 2>(a, st, dev.device, dev.num_sms, dev.max_smem_optin)
                 : gemv_dispatch<false, true, 2>(a, st, dev.device, dev.num_sms, dev.max_smem_optin);
    return z ? gemv_dispatch<false, false, 4>(a, st, dev.device, dev.num_sms, dev.max_smem_optin)
             : gemv_dispatch<false, true, 4>(a, st, dev.device, dev.num_sms, dev.max_smem_optin);
}

}  // namespace w4
