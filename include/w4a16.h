/*
 * w4a16.h -- C ABI of the fused 4-bit-weight x BF16-activation kernels for
 * NVIDIA GB300 (sm_103a).
 *
 * Operation (problem statement of the pages; "Lab 5: Gemma4 end-to-end
 * inference optimisation", sections "INT4 fused GEMV" and "Final
 * configuration"; "DeepSeek V4 Triton FP4 optimisation in practice", deep
 * analysis item 2):
 *
 *     Y[m, n] = sum_k X[m, k] * W[n, k]            (Y = X * W^T)
 *     INT4:  W[n, k] = (q[n, k] - z[n, k/g]) * s[n, k/g],  g = 128
 *     FP4:   W[n, k] = e2m1(q[n, k]) * s[n, k/g],           g = 32
 *
 * with q a 4-bit code packed two per byte along K: byte n*(K/2) + k/2 holds
 * column k in its low nibble when k is even and in its high nibble when k is
 * odd.  s and z are IEEE binary16, X and Y bfloat16 (passed as raw 16-bit
 * patterns in uint16_t buffers), all row-major and contiguous.  e2m1 is the
 * OCP MX FP4 format (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives).
 * Products accumulate in binary32; outputs are rounded to bfloat16 with
 * round-to-nearest-even.  No dequantised weight is written to memory except
 * by the debug entry w4a16_dequant.
 *
 * Conventions shared by every entry point:
 *  - all data pointers are DEVICE pointers owned by the caller; the library
 *    keeps no reference after the call returns and allocates no memory;
 *  - kernels run on the CURRENT device (cudaSetDevice) and every data
 *    pointer must be memory of that device (device memory of it, or managed
 *    memory): a pointer to another device's memory or to host memory is
 *    refused with W4A16_ERR_INVALID_ARG before anything is launched (the
 *    one exception: w4a16_copy also takes pinned, mapped host memory);
 *  - every data pointer must be 16-byte aligned (else W4A16_ERR_MISALIGNED);
 *  - an output must not overlap any input of the same call (CTAs write
 *    their outputs while others may still read the inputs); this is not
 *    checked;
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream); calls are
 *    asynchronous on it and never synchronise the host, so they may be
 *    captured into a CUDA graph;
 *  - arguments are checked on the host before anything is launched; a failed
 *    check launches nothing and returns a nonzero w4a16_status, with a
 *    message available from w4a16_last_error_string();
 *  - kernels never trap: a device-side problem (an expert id out of range, a
 *    pipeline wait that timed out) sets a sticky per-device status word that
 *    w4a16_check_device_error() reports and clears.  There is one status
 *    word per device, shared by the launches of every stream and host thread
 *    on that device.
 *  - host threads may call concurrently (the per-device set-up made on first
 *    use is guarded); the usual rule holds that concurrent calls on one
 *    stream are ordered as the host makes them.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad enum  */
    W4A16_ERR_UNSUPPORTED = 2,  /* valid but not implemented (group, K range) */
    W4A16_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned           */
    W4A16_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed       */
    W4A16_ERR_TIMEOUT = 5,      /* a device pipeline wait gave up             */
    W4A16_ERR_DEVICE = 6        /* a device-side data error (bad expert id)   */
} w4a16_status;

typedef enum { W4_FMT_INT4_ASYM = 0, W4_FMT_FP4_E2M1 = 1 } w4_format;
typedef enum { W4_OUT_F32 = 0, W4_OUT_BF16 = 1 } w4_out_dtype;

/*
 * Decode GEMV, M = 1 ("Lab 5", section "INT4 fused GEMV": the decode linear
 * reads the packed INT4 weight once, unpacks it in registers, applies the
 * per-group scale and zero and dots it with the activation vector).
 *   x  : bfloat16 [K]          activation
 *   qw : uint8    [N, K/2]     packed INT4 codes
 *   s  : binary16 [N, K/group] scales
 *   z  : binary16 [N, K/group] zero points, or NULL for symmetric INT4:
 *        the zero point is then the code midpoint 8 for every group ("Lab 5",
 *        section "Quantisation correctness": the symmetric GPTQ variant)
 *   y  : bfloat16 [N]          output (overwritten)
 * Requires group == 128, N >= 1, 128 <= K <= 16384, K % 128 == 0.
 */
int w4a16_gemv(const uint16_t *x, const uint8_t *qw, const uint16_t *s,
               const uint16_t *z, uint16_t *y, int64_t N, int64_t K,
               int group, void *stream);

/*
 * Prefill GEMM, M >= 1 ("Lab 5", sections "Triton dequant + cuBLAS" and
 * "INT4 fused GEMV", M = 128 prefill check; here fused: weight tiles are
 * dequantised into shared memory and fed to the tcgen05 tensor cores, so no
 * BF16 weight matrix is written to HBM).
 *   X : bfloat16 [M, K];  qw, s, z as for w4a16_gemv (z may be NULL:
 *       symmetric INT4);  Y : bfloat16 [M, N].
 * Requires group == 128, K % 128 == 0, 128 <= K <= 16384, N >= 1.  Any
 * M >= 1 and any N are accepted (rows past M and N in the last tiles are
 * masked).  Decode-sized
 * batches run as the streaming GEMV instead: M <= 4 rows share one pass over
 * the weights (two passes of two rows where K leaves fewer teams per CTA);
 * larger M runs on the tensor cores.
 */
int w4a16_gemm(const uint16_t *X, const uint8_t *qw, const uint16_t *s,
               const uint16_t *z, uint16_t *Y, int64_t M, int64_t N,
               int64_t K, int group, void *stream);

/*
 * The prefill GEMM of w4a16_gemm with binary16 operands ("Lab 5", section
 * "Triton dequant + cuBLAS": the same product; here the weights are
 * dequantised once per tile and never written to HBM):
 *  - a pre-pass scales each row of X by a power of two into binary16 (every
 *    value within 2^28 of the row's largest magnitude exact; the epilogue
 *    undoes the scale);
 *  - each weight is formed as fl16(fl16(q - z) * s): one rounding when z is
 *    an integer, a relative error of at most 2^-11 (the BF16 weights of the
 *    dequantise-then-GEMM path carry 2^-9);
 *  - one binary32 accumulator runs over all of K, on tiles of 128 weight
 *    rows x 256 token rows.
 * So |Y - X W^T| <= 2^-10 sum_k |X[m,k] W[n,k]| plus the BF16 rounding of
 * the output.  w4a16_gemm is exact in every product (the scale is applied
 * per group to binary32 partial sums), which keeps outputs that cancel
 * exact when activations carry outliers far above the rest; this entry is
 * the faster one from M = 256 on.
 * Layouts and requirements: those of w4a16_gemm (any M >= 1, any N).
 * Scratch: M*K*2 + 4*M bytes, stream-ordered, from a memory pool that the
 * library keeps per device (kept reserved between calls); under stream
 * capture it becomes an allocation of the CUDA graph.
 */
int w4a16_gemm_f16(const uint16_t *X, const uint8_t *qw, const uint16_t *s,
                   const uint16_t *z, uint16_t *Y, int64_t M, int64_t N,
                   int64_t K, int group, void *stream);

/*
 * Dense BF16 GEMM, Y[m, n] = sum_k X[m, k] * W[n, k] on the tensor cores:
 * the second pass of the unfused path ("Lab 5", section "Triton dequant +
 * cuBLAS": dequantise to a BF16 weight matrix in memory, then a dense GEMM).
 * With w4a16_dequant (W4_OUT_BF16) it forms the two-pass ablation of the
 * fused w4a16_gemm, measuring what the fusion saves.
 *   X : bfloat16 [M, K];  W : bfloat16 [N, K];  Y : bfloat16 [M, N]
 *       (binary32 accumulation, round-to-nearest-even output).
 * Requires K % 64 == 0, M, N >= 1.
 */
int w4a16_bf16_gemm(const uint16_t *X, const uint16_t *W, uint16_t *Y,
                    int64_t M, int64_t N, int64_t K, void *stream);

/*
 * Copy `bytes` bytes from src to dst with one kernel on `stream`, launched
 * with programmatic dependent launch: the small transfers of a decode step
 * ("Lab 5: Gemma4 end-to-end inference optimisation", section "CUDA Graph":
 * the step's launches captured and replayed as one graph) -- the token's
 * activation in, the step's result out -- then chain with the library's
 * kernels instead of being copy-engine operations between them.
 *   dst, src : memory of the current device, managed memory, or PINNED host
 *              memory mapped into the device's address space (cudaHostAlloc
 *              or cudaHostRegister with mapping, which unified addressing
 *              gives by default); this is the one entry point that takes
 *              host pointers.  Any alignment (16-byte moves when both are
 *              16-byte aligned); the ranges must not overlap.
 *   bytes    : >= 0 (0 launches nothing and accepts null pointers).
 * Pageable host memory, pinned host memory without a device mapping and
 * another device's memory are refused with W4A16_ERR_INVALID_ARG before
 * anything is launched.  The host may read a pinned destination once the
 * stream has been synchronised.
 */
int w4a16_copy(void *dst, const void *src, int64_t bytes, void *stream);

/*
 * Batched-expert FP4 GEMV for one token ("DeepSeek V4 Triton FP4
 * optimisation in practice": six routed experts per token; stacking the
 * experts on the host cost 20% end to end, so all experts run in one launch
 * reading the expert weights in place).
 *   x          : bfloat16 [K]
 *   qw         : uint8    [E, N, K/2]     packed E2M1 codes of every expert
 *   s          : binary16 [E, N, K/group] scales
 *   expert_ids : int32    [topk]          DEVICE array; row i of y uses
 *                                         expert expert_ids[i]; repeats allowed
 *   y          : bfloat16 [topk, N]
 * Requires group == 32, K % 64 == 0, 64 <= K <= 16384, 1 <= topk.
 * An id outside [0, E) cannot be checked on the host: that output row is
 * written as zeros and the device status is set (W4A16_ERR_DEVICE).
 */
int fp4_moe_gemv(const uint16_t *x, const uint8_t *qw, const uint16_t *s,
                 const int32_t *expert_ids, int topk, uint16_t *y, int64_t E,
                 int64_t N, int64_t K, int group, void *stream);

/*
 * Batched-expert FP4 GEMM for M tokens, each routed to topk experts
 * ("DeepSeek V4 Triton FP4 optimisation in practice": the fused FP4
 * dequantise-and-multiply expert GEMMs; M > 1 is the prefill or batched
 * decode case of the one-token fp4_moe_gemv):
 *   Y[m, j, n] = sum_k X[m, k] * e2m1(qw[e, n, k]) * s[e, n, k/32],
 *   e = expert_ids[m * topk + j].
 *   X          : bfloat16 [M, K]
 *   qw         : uint8    [E, N, K/2]     packed E2M1 codes (even k in the
 *                                         low nibble) of every expert
 *   s          : binary16 [E, N, K/group] scales
 *   expert_ids : int32    [M, topk]       DEVICE array; repeats allowed
 *   Y          : bfloat16 [M, topk, N]
 *   scratch    : device memory of at least fp4_moe_gemm_scratch_bytes(M,
 *                topk, E, K) bytes, 256-byte aligned, owned by the caller and
 *                used by this call only while it runs on `stream` (the
 *                routing table and the tokens gathered per expert); it need
 *                not be zeroed.
 * Three launches on `stream`: routing, gathering, the tensor-core GEMM (they
 * can be captured in a CUDA graph; each replay routes the ids it finds).
 * Arithmetic: each weight e2m1 * s is rounded once to binary16 (relative
 * error at most 2^-11 for |s| in [2^-13, 10922]; smaller scales round to
 * binary16 subnormals, larger ones overflow); each token row is scaled by
 * a power of two into binary16 (exact for values within 2^28 of its
 * largest magnitude); products and sums in binary32; output rounded to
 * nearest even.  fp4_moe_gemv applies the scales in binary32 instead and
 * has no range limit on s.
 * Requires group == 32, K % 256 == 0, K <= 65536, M * topk <= 2^20,
 * E <= 8192.  An id outside [0, E) cannot be checked on the host: that
 * output row is written as zeros and the device status is set
 * (W4A16_ERR_DEVICE).
 */
int fp4_moe_gemm(const uint16_t *X, const uint8_t *qw, const uint16_t *s,
                 const int32_t *expert_ids, int M, int topk, uint16_t *Y,
                 int64_t E, int64_t N, int64_t K, int group, void *scratch,
                 int64_t scratch_bytes, void *stream);

/* Scratch bytes fp4_moe_gemm needs (0 for sizes below 1). */
int64_t fp4_moe_gemm_scratch_bytes(int M, int topk, int64_t E, int64_t K);

/*
 * Debug dequantisation: writes the dequantised weight matrix (the step the
 * fused kernels keep in registers / shared memory; "Lab 5", section "Triton
 * dequant + cuBLAS", first pass).  Bit-exact contract:
 *   INT4: W = fl32(fl32((float)q - (float)z) * (float)s)
 *   FP4 : W = fl32(e2m1(q) * (float)s)           (exact)
 *   out_dtype W4_OUT_F32 writes binary32, W4_OUT_BF16 writes
 *   round-to-nearest-even bfloat16 of that binary32 value.
 *   qw : uint8 [rows, K/2];  s (and z for INT4) binary16 [rows, K/group];
 *   z must be NULL for FP4; for INT4 a NULL z means symmetric INT4 (z = 8);
 *   out : [rows, K] binary32 or bfloat16.
 * group must be 128 (INT4) or 32 (FP4); K % group == 0; rows >= 1.
 */
int w4a16_dequant(int fmt, const uint8_t *qw, const uint16_t *s,
                  const uint16_t *z, void *out, int out_dtype, int64_t rows,
                  int64_t K, int group, void *stream);

/*
 * One INT4 linear of a decode sequence: Y = X W^T exactly as w4a16_gemm
 * computes it (M = 1 as w4a16_gemv), with the same layouts.
 *   x  : bfloat16 [M, K];  qw : uint8 [N, K/2];  s : binary16 [N, K/group];
 *   z  : binary16 [N, K/group] or NULL (symmetric INT4);  y : bfloat16 [M, N].
 * Requirements: those of w4a16_gemv when M == 1, of w4a16_gemm when M > 1.
 */
typedef struct {
    const uint16_t *x;
    const uint8_t *qw;
    const uint16_t *s;
    const uint16_t *z;
    uint16_t *y;
    int64_t M, N, K;
} w4a16_linear;

/*
 * A decode step as one call ("Lab 5", sections "CUDA Graph" and
 * "Performance analysis": a decode step is 328 quantised linears plus the
 * vocabulary GEMV, and the launch overhead of the short GEMVs is what the
 * CUDA graph removes).  Launches ops[0 .. count-1] in order on `stream`.
 * Each op reads its x and writes its y only after the previous op has
 * finished (only its weight prefetch into L2 may overlap the previous op),
 * so an op may read the output of any earlier op and may overwrite a buffer
 * that an earlier op read (but, as for every call, not its own input).  The
 * `ops` array is read during the call only.
 * Every op is checked before anything is launched: a failed check launches
 * nothing and the message names the op.  count == 0 launches nothing and
 * returns W4A16_OK.  A CUDA launch error at op i returns W4A16_ERR_CUDA
 * with ops 0 .. i-1 already queued.
 */
int w4a16_linear_sequence(const w4a16_linear *ops, int count, int group,
                          void *stream);

/*
 * A chain of M = 1 INT4 linears in ONE persistent launch ("Lab 5", sections
 * "CUDA Graph" and "Performance analysis": a decode step is 328 short
 * bandwidth-bound GEMVs plus the vocabulary GEMV, and what separates them --
 * launch overhead, each grid's ramp and drain -- is time the step loses).
 * Computes what w4a16_linear_sequence computes for the same ops, with the
 * same results bit for bit: each op reads its x only after every earlier op
 * that writes it has finished, and writes its y only after every earlier op
 * that reads or writes it has finished.  The packed weights of later ops
 * stream into shared memory while earlier ops finish, so ops must not write
 * any op's weights (refused).  Every op must have M == 1 (else
 * W4A16_ERR_UNSUPPORTED) and pass the checks of w4a16_gemv; an op whose y
 * overlaps its own x is refused.  The dependencies are found on the host
 * from the address ranges of x and y.  Ops are launched in pieces of up to
 * 192 per kernel (a dependency across pieces is met by the stream order).
 *   scratch       : device memory of at least
 *                   w4a16_linear_chain_scratch_bytes(count) bytes, 4-byte
 *                   aligned, caller-owned, ALL ZERO before its first use
 *                   (cudaMemset); the kernel keeps one completion counter per
 *                   op there and every call leaves it all zero again (also
 *                   one whose waits timed out), so the next call on the same
 *                   stream may reuse it as is.  Calls that may run at the
 *                   same time (other streams) need separate scratch.
 *   scratch_bytes : its size in bytes.
 * One CTA per SM; a launch in which some op depends on another is
 * cooperative (all CTAs resident at once).  count == 0 launches nothing.
 */
int64_t w4a16_linear_chain_scratch_bytes(int count);
int w4a16_linear_chain(const w4a16_linear *ops, int count, int group,
                       void *scratch, int64_t scratch_bytes, void *stream);

/*
 * w4a16_linear_chain without caller scratch: the same computation, for
 * callers that cannot allocate device memory of their own -- for instance an
 * engine that hands every byte of the GPU to its own memory pool and gives
 * plug-in code only the tensors it works on, or code that must not call
 * cudaMalloc because of the device-wide synchronisation it can cause.  (The
 * pages have no counterpart: this is an interface choice of this library.)
 * The per-linear completion counters live in a 16 KB array that the library
 * holds on every device that loads it, until the library is unloaded; this
 * call allocates nothing.
 *   Limit: at most 4032 linears per call (W4A16_ERR_UNSUPPORTED beyond).
 *   The first call on a device looks up the array's device address (once
 *   per device); make that first call before any stream capture.
 *   Every call clears the counters it uses (a memset on `stream`) before its
 *   launches.  All calls on a device share the one array: two calls whose
 *   work can overlap on the GPU (different streams without ordering between
 *   them) race on it and may compute wrong results or time out; serialise
 *   them (one stream, or events).
 * ops, count, group and stream are as for w4a16_linear_chain.
 */
int w4a16_linear_chain_noalloc(const w4a16_linear *ops, int count, int group,
                               void *stream);

/*
 * The same sequence captured once into a CUDA graph and replayed by
 * w4a16_graph_launch: one host call per decode step, with the launches
 * chained on the device.
 *   w4a16_graph_create  checks every op as w4a16_linear_sequence does (a
 *       failed check captures nothing), captures the launches on a private
 *       stream of the current device, instantiates the graph and returns an
 *       opaque handle in *out (NULL on any failure; count must be >= 1).
 *       The graph keeps the ops' pointers, not their contents: every buffer
 *       must stay allocated at the same address until the handle is
 *       destroyed, and each replay reads the buffers as they are when it
 *       runs (write the next step's x in place between replays).  The
 *       injection flags in force at creation are kept by the graph.
 *   w4a16_graph_launch  enqueues one replay on `stream` (a stream of the
 *       device the graph was created on); asynchronous like every call.
 *   w4a16_graph_destroy releases the handle (NULL is accepted); a replay
 *       still in flight completes first.
 * The handle is owned by the caller and may be used from one host thread at
 * a time.
 */
typedef struct w4a16_graph_s *w4a16_graph_t;
int w4a16_graph_create(const w4a16_linear *ops, int count, int group,
                       w4a16_graph_t *out);
int w4a16_graph_launch(w4a16_graph_t graph, void *stream);
int w4a16_graph_destroy(w4a16_graph_t graph);

/*
 * Synchronises `stream`, then reads and clears the current device's sticky
 * status.  Returns W4A16_OK, W4A16_ERR_TIMEOUT, W4A16_ERR_DEVICE or
 * W4A16_ERR_CUDA.  The status word is per device, not per stream: only
 * `stream` is synchronised, so a bit set by a launch on another stream that
 * is still running may be missed, and a bit set by another stream's launch
 * is reported (and cleared) here.  Synchronise the device first (or use one
 * stream) to attribute the status to particular launches.
 */
int w4a16_check_device_error(void *stream);

/*
 * Test-only failure injection (the library's bounded-wait path, exercised
 * without faulting the GPU).  Sets this device's injection flags:
 *   0  normal operation;
 *   1  every later w4a16_gemv, fp4_moe_gemv and w4a16_gemm launch issues no
 *      stage of its pipeline (the weight stages of the GEMVs, the activation
 *      stages of the GEMM), so its waits run out after their limit (about
 *      2 s); the launch then returns with an unspecified output and
 *      w4a16_check_device_error reports W4A16_ERR_TIMEOUT (the context stays
 *      usable);
 *   2  the same launches issue their pipeline stages but never consume
 *      them, so the producers' waits for free stages run out while their
 *      copies are issued: each producer then waits for its own copies to
 *      land before the launch ends (W4A16_ERR_TIMEOUT as for flag 1).
 * The flags are a host-side setting passed to each later launch (a CUDA
 * graph keeps the flags it was captured with).  Not for production use.
 * Returns W4A16_OK, or W4A16_ERR_INVALID_ARG for an unknown flag.
 */
int w4a16_debug_inject(unsigned int flags);

/* Message for the last failed call on this host thread ("" if none). */
const char *w4a16_last_error_string(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int w4a16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
