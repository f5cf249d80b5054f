// Dense BF16 GEMM on the tcgen05 tensor cores, Y[m, n] = sum_k X[m, k] W[n, k]:
// the second pass of the unfused path ("Lab 5: Gemma4 end-to-end inference
// optimisation", section "Triton dequant + cuBLAS": a dequantiser writes the
// BF16 weight matrix to memory, then a dense BF16 GEMM reads it back).  With
// w4a16_dequant it forms the two-pass ablation of the fused w4a16_gemm.
//
// One CTA computes a tile of 128 weight rows n x 128 activation rows m over
// the whole of K into one tensor-memory accumulator (128 lanes = n,
// 128 columns = m):
//  * warp 0 (one lane): per 64-wide K block, one TMA box of W (128 rows x
//    128 bytes) and one of X, 128-byte swizzle, into a ring of stages;
//  * warp 1 (one lane): allocates tensor memory, per stage waits for it,
//    issues 4 x tcgen05.mma (M=128, N=128, K=16; A = W and B = X, both from
//    shared memory) and commits to the stage's "empty" barrier; after the
//    last stage it commits to the accumulator barrier;
//  * warps 4-7: read the accumulator (warp w: TMEM lanes 32 (w mod 4) .. +31),
//    round to BF16 and store Y.
// Every wait is bounded; on timeout the status word is set and each role
// still performs the arrivals the others wait for.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace w4 {
namespace {

constexpr int TN = 128;                 // weight rows per tile (the MMA's M)
constexpr int TM = 128;                 // activation rows per tile (the MMA's N)
constexpr int BK = 64;                  // K per stage: one 128-byte swizzled box row
constexpr int BOX_BYTES = 128 * 128;    // 16 KB: 128 rows x 128 bytes
constexpr int STAGE_BYTES = 2 * BOX_BYTES;
constexpr int STAGES = 6;
constexpr int THREADS = 256;            // warps 0, 1: producer, MMA; 4-7: epilogue
constexpr uint32_t TMEM_COLS = 128;

struct DenseArgs {
    uint16_t *Y;
    unsigned int *status;
    int M, N, K;
};

struct DenseBarriers {
    uint64_t full[STAGES];   // both boxes of the stage landed (TMA tx bytes)
    uint64_t empty[STAGES];  // MMAs done with the stage (commit)
    uint64_t accfull;        // accumulator complete (commit)
    uint32_t tmem_holder;
};

__global__ void __launch_bounds__(THREADS, 1)
bf16_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const DenseArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    DenseBarriers &bar = *reinterpret_cast<DenseBarriers *>(smem + STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * TN;
    const int m0 = blockIdx.y * TM;
    const int nk = a.K / BK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&bar.full[i], 1);
            mbar_init(&bar.empty[i], 1);
        }
        mbar_init(&bar.accfull, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&bar.tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_holder;
    // programmatic dependent launch: this grid may start while the previous
    // launch of the stream finishes; every global read and write follows
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmW);
            tma_prefetch_desc(&tmX);
            for (int kb = 0; kb < nk; ++kb) {
                const int st = kb % STAGES;
                if (kb >= STAGES && !mbar_wait(&bar.empty[st], ((kb / STAGES) - 1) & 1, a.status)) break;
                unsigned char *dst = smem + st * STAGE_BYTES;
                mbar_arrive_expect_tx(&bar.full[st], STAGE_BYTES);
                // rows past N or M (tile tails) read as zeros
                tma_load_2d(dst, &tmW, kb * BK, n0, &bar.full[st]);
                tma_load_2d(dst + BOX_BYTES, &tmX, kb * BK, m0, &bar.full[st]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_kind_f16(TN, TM, 1u);  // BF16 x BF16 -> F32
        int kb = 0;
        for (; kb < nk; ++kb) {
            const int st = kb % STAGES;
            if (!mbar_wait(&bar.full[st], (kb / STAGES) & 1, a.status)) break;
            tc_fence_after();
            {
                const uint32_t a_addr = smem_u32(smem + st * STAGE_BYTES);
                const uint32_t b_addr = a_addr + BOX_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_f16_w(tmem, smem_desc_sw128_kmajor(a_addr + 32 * k), smem_desc_sw128_kmajor(b_addr + 32 * k),
                               idesc, (kb | k) != 0);
                umma_commit_w(&bar.empty[st]);
            }
            __syncwarp();
        }
        // the accumulator barrier fires once every MMA issued has completed
        // (also after a timeout, so that the epilogue's wait ends); MMAs
        // always complete, so this warp waits for it ignoring the status
        // word: tensor memory is never released under an MMA in flight
        umma_commit_w(&bar.accfull);
        __syncwarp();
        mbar_wait(&bar.accfull, 0, nullptr);
    } else if (warp >= 4) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int n = n0 + q * 32 + lane;  // output column of this thread
        const bool ok = mbar_wait_lanes(lane == 0 ? &bar.accfull : nullptr, 0, a.status);
        tc_fence_after();
        if (ok) {
            const uint32_t t_acc = tmem + (static_cast<uint32_t>(q * 32) << 16);
            const int mrows = min(TM, a.M - m0);
#pragma unroll
            for (int c = 0; c < TM / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_acc + 32 * c, r);
                tmem_ld_wait();
                if (n < a.N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (32 * c + j < mrows)
                            a.Y[static_cast<size_t>(m0 + 32 * c + j) * a.N + n] = f32_to_bf16_bits(__uint_as_float(r[j]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_bf16_gemm(const uint16_t *X, const uint16_t *W, uint16_t *Y, int64_t M, int64_t N, int64_t K,
                             cudaStream_t st, unsigned int *status, const DeviceInfo &dev) {
    CUtensorMap tmW, tmX;
    // W bf16 [N, K] and X bf16 [M, K]: boxes of 64 K x 128 rows, 128-byte swizzle
    if (!encode_2d_sw128(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, static_cast<uint64_t>(N),
                         static_cast<uint64_t>(K), static_cast<uint64_t>(K) * 2, BK, TN) ||
        !encode_2d_sw128(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, static_cast<uint64_t>(M),
                         static_cast<uint64_t>(K), static_cast<uint64_t>(K) * 2, BK, TM))
        return cudaErrorInvalidValue;
    DenseArgs a;
    a.Y = Y;
    a.status = status;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    const int smem = 1024 + STAGES * STAGE_BYTES + static_cast<int>(sizeof(DenseBarriers));
    if (smem > dev.max_smem_optin) return cudaErrorNotSupported;
    static SmemLimit limit;
    if (cudaError_t e = limit.ensure(reinterpret_cast<const void *>(bf16_gemm_tc_kernel), dev.device, smem)) return e;
    const dim3 grid(static_cast<unsigned>((N + TN - 1) / TN), static_cast<unsigned>((M + TM - 1) / TM), 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bf16_gemm_tc_kernel, tmW, tmX, a);
}

}  // namespace w4
