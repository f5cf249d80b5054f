/*
 * w4a16 oracle: plain, slow, obviously correct CPU reference for the fused
 * 4-bit-weight x BF16-activation products.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library and includes none of it.
 *
 * Sources (page titles as published):
 *  [Lab5]  "Lab 5: Gemma4 end-to-end inference optimisation" (docs.bfyes.cn,
 *          study/hpc/lab5), sections "Quantisation correctness" (GPTQ INT4,
 *          group 128, asymmetric, FP16 scale), "INT4 fused GEMV" (read packed
 *          INT4, unpack, apply the per-group scale/zero, dot with the input)
 *          and "Final configuration" (config.yaml quantisation keys).
 *  [DSV4]  "DeepSeek V4 Triton FP4 optimisation in practice" (ai-engineering
 *          pages, Ch01.377), "Deep analysis" item 2: even K columns pair with
 *          the low nibble, odd K columns with the high nibble.
 *  The problem statement fixes the remaining arithmetic:
 *          y[m,n] = sum_k x[m,k] * W[n,k],  W[n,k] = (q[n,k] - z[n,k/g]) * s[n,k/g]
 *          with q packed two per byte along K, low nibble = even k, s and z FP16.
 *  Symmetric INT4 ([Lab5] "Quantisation correctness": symmetric GPTQ is the
 *  variant the lab measured before settling on asymmetric) is taken in its
 *  GPTQ form, the zero point being the code midpoint 2^(4-1) = 8: it is the
 *  asymmetric formula with z = 8, selected by passing z = NULL.
 *  FP4 E2M1 values follow the OCP Microscaling (MX) format definition
 *  (1 sign, 2 exponent bits with bias 1, 1 mantissa bit, no inf/NaN); the
 *  pages name the format but print no table.
 *
 * Arithmetic contract (kept deliberately simple):
 *  - dequantised weights are formed in binary32 exactly as two rounded
 *    operations, (float)q - (float)z, then * (float)s, with FP contraction
 *    disabled at compile time (-ffp-contract=off);
 *  - products and sums are taken in binary64 with k ascending;
 *  - results are returned in binary64; rounding to BF16 is a separate,
 *    explicit round-to-nearest-even step.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

/* Threads for the products below (1 unless oracle_set_threads raises it).
 * Each output element is computed by one thread exactly as in the serial
 * loop (same operations, k ascending), so the results do not depend on the
 * thread count; only the timed CPU baseline uses more than one. */
static int g_threads = 1;

void oracle_set_threads(int n)
{
    g_threads = n < 1 ? 1 : n;
}

/* ---------------------------------------------------------------- formats */

/* IEEE 754 binary16 bit pattern -> value (format definition). */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);  /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 bit pattern -> value: bfloat16 is the upper half of binary32. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary64 -> bfloat16 bit pattern, round to nearest, ties to even, taken in
 * one step from the binary64 value (no intermediate binary32 rounding). */
uint16_t oracle_f64_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v))
        return (uint16_t)(sign | 0x7fc0u);
    if (isinf(a))
        return (uint16_t)(sign | 0x7f80u);
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);                /* a = f * 2^e, f in [0.5, 1) */
    /* bfloat16 keeps 8 significant bits; below 2^-126 the quantum is 2^-133. */
    int q_exp = (e - 1 >= -126) ? (e - 8) : -133;
    double q = rint(ldexp(a, -q_exp)); /* default rounding mode: ties to even */
    double r = ldexp(q, q_exp);        /* exact */
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7f80u);
    /* r is exactly representable in binary32 and in bfloat16 */
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7fffu));
}

/* Round each binary64 value to a bfloat16 bit pattern. */
void oracle_round_bf16(const double *y, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f64_to_bf16(y[i]);
}

/* --------------------------------------------------------------- unpacking */

/* The 4-bit code of element (n, k) of a row-major packed matrix with K codes
 * per row: byte n*(K/2) + k/2, low nibble for even k, high nibble for odd k
 * ([DSV4] deep analysis 2; problem statement). */
int oracle_code(const uint8_t *qw, int64_t K, int64_t n, int64_t k)
{
    uint8_t b = qw[n * (K / 2) + k / 2];
    return (k % 2 == 0) ? (b & 0x0f) : (b >> 4);
}

/* E2M1 code -> value (OCP MX): sign bit 3, exponent bits 2..1 (bias 1),
 * mantissa bit 0; exponent 0 is subnormal (0 or 0.5). */
double oracle_e2m1_value(int code)
{
    int sign = (code >> 3) & 1;
    int ex = (code >> 1) & 3;
    int m = code & 1;
    double mag = (ex == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, ex - 1);
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------- dequantise */

/* INT4 asymmetric group dequantisation ([Lab5] quantisation correctness and
 * final configuration: bits 4, group_size g, symmetric false, FP16 scale;
 * problem statement: W = (q - z) * s).  One binary32 value per element:
 * (float)q - (float)z rounded, then times (float)s rounded.
 * qw: [N, K/2] bytes; s, z: [N, K/g] binary16; W: [N, K] binary32.
 * z == NULL: symmetric INT4, z = 8 for every group. */
void oracle_dequant_int4(const uint8_t *qw, const uint16_t *s, const uint16_t *z,
                         int64_t N, int64_t K, int64_t g, float *W)
{
    int64_t G = K / g;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            float q = (float)oracle_code(qw, K, n, k);
            float zf = z ? (float)oracle_f16_to_f64(z[n * G + k / g]) : 8.0f;
            float sf = (float)oracle_f16_to_f64(s[n * G + k / g]);
            float d = q - zf;
            float w = d * sf;
            W[n * K + k] = w;
        }
    }
}

/* FP4 E2M1 dequantisation with one binary16 scale per g codes along K
 * ([DSV4] "FP4 packed -> BF16" dequant path; scale layout from the problem
 * statement).  rows = E*N for a stack of experts.  W = e2m1(code) * s in
 * binary32 (exact: at most 2 + 11 significant bits). */
void oracle_dequant_fp4(const uint8_t *qw, const uint16_t *s, int64_t rows,
                        int64_t K, int64_t g, float *W)
{
    int64_t G = K / g;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t k = 0; k < K; ++k) {
            float v = (float)oracle_e2m1_value(oracle_code(qw, K, r, k));
            float sf = (float)oracle_f16_to_f64(s[r * G + k / g]);
            W[r * K + k] = v * sf;
        }
    }
}

/* ------------------------------------------------------------- products */

/* y[m, n] = sum_k x[m, k] * W[n, k] for INT4 weights ([Lab5] INT4 fused GEMV:
 * the weight is dequantised per element and dotted with the activation;
 * M = 1 is the decode GEMV, M > 1 the prefill GEMM).  Each W[n,k] is the
 * binary32 value of oracle_dequant_int4; the product and the running sum are
 * binary64, k ascending.  X: [M, K] bfloat16; Y: [M, N] binary64.
 * z == NULL: symmetric INT4 (z = 8), as in oracle_dequant_int4. */
void oracle_gemm_int4(const uint16_t *X, const uint8_t *qw, const uint16_t *s,
                      const uint16_t *z, int64_t M, int64_t N, int64_t K,
                      int64_t g, double *Y)
{
    int64_t G = K / g;
#pragma omp parallel for collapse(2) schedule(static) num_threads(g_threads) if (g_threads > 1)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                float q = (float)oracle_code(qw, K, n, k);
                float zf = z ? (float)oracle_f16_to_f64(z[n * G + k / g]) : 8.0f;
                float sf = (float)oracle_f16_to_f64(s[n * G + k / g]);
                float d = q - zf;
                float w = d * sf;
                acc += (double)w * oracle_bf16_to_f64(X[m * K + k]);
            }
            Y[m * N + n] = acc;
        }
    }
}

/* Batched-expert FP4 GEMV ([DSV4] core insight on stacking overhead and deep
 * analysis 4: six routed experts per token, each a separate weight matrix).
 * Output row i uses expert ids[i]: y[i, n] = sum_k x[k] * W_{ids[i]}[n, k],
 * with W_e the binary32 values of oracle_dequant_fp4 on expert e's slice.
 * qw: [E, N, K/2]; s: [E, N, K/g]; x: [K] bfloat16; Y: [topk, N] binary64.
 * An id outside [0, E) gives a zero row and increments *bad. */
void oracle_moe_fp4(const uint16_t *x, const uint8_t *qw, const uint16_t *s,
                    const int32_t *ids, int64_t topk, int64_t E, int64_t N,
                    int64_t K, int64_t g, double *Y, int *bad)
{
    int64_t G = K / g;
    for (int64_t i = 0; i < topk; ++i) {
        int64_t e = ids[i];
        if (e < 0 || e >= E) {
            for (int64_t n = 0; n < N; ++n)
                Y[i * N + n] = 0.0;
            if (bad)
                *bad += 1;
            continue;
        }
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1)
        for (int64_t n = 0; n < N; ++n) {
            int64_t r = e * N + n;   /* row of the [E*N, K] stack */
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                float v = (float)oracle_e2m1_value(oracle_code(qw, K, r, k));
                float sf = (float)oracle_f16_to_f64(s[r * G + k / g]);
                float w = v * sf;
                acc += (double)w * oracle_bf16_to_f64(x[k]);
            }
            Y[i * N + n] = acc;
        }
    }
}

/* Batched-expert FP4 GEMM for M tokens ([DSV4] the fused FP4 expert GEMMs:
 * every token is routed to topk experts, each a separate weight matrix; M > 1
 * is the prefill / batched case).  Output row (m, j) uses expert
 * ids[m*topk + j]: y[m, j, n] = sum_k X[m, k] * W_{ids[m*topk+j]}[n, k], with
 * W_e the binary32 values of oracle_dequant_fp4 on expert e's slice, every
 * product and the running sum in binary64, k ascending.
 * X: [M, K] bfloat16; ids: [M, topk]; qw: [E, N, K/2]; s: [E, N, K/g];
 * Y: [M, topk, N] binary64.  An id outside [0, E) gives a zero row and
 * increments *bad. */
void oracle_moe_fp4_gemm(const uint16_t *X, const uint8_t *qw, const uint16_t *s,
                         const int32_t *ids, int64_t M, int64_t topk, int64_t E,
                         int64_t N, int64_t K, int64_t g, double *Y, int *bad)
{
    int64_t G = K / g;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = 0; j < topk; ++j) {
            int64_t e = ids[m * topk + j];
            double *y = Y + (m * topk + j) * N;
            if (e < 0 || e >= E) {
                for (int64_t n = 0; n < N; ++n)
                    y[n] = 0.0;
                if (bad)
                    *bad += 1;
                continue;
            }
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1)
            for (int64_t n = 0; n < N; ++n) {
                int64_t r = e * N + n;   /* row of the [E*N, K] stack */
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    float v = (float)oracle_e2m1_value(oracle_code(qw, K, r, k));
                    float sf = (float)oracle_f16_to_f64(s[r * G + k / g]);
                    float w = v * sf;
                    acc += (double)w * oracle_bf16_to_f64(X[m * K + k]);
                }
                y[n] = acc;
            }
        }
    }
}

/* ---------------------------------------------------- two-pass ablation */

/* Dense product of bfloat16 matrices, the second pass of the unfused path
 * ([Lab5] "Triton dequant + cuBLAS": dequantise to a BF16 weight matrix in
 * memory, then a dense BF16 GEMM): Y[m, n] = sum_k X[m, k] * W[n, k], every
 * product and the running sum in binary64, k ascending.
 * X: [M, K] bfloat16; W: [N, K] bfloat16; Y: [M, N] binary64. */
void oracle_gemm_bf16(const uint16_t *X, const uint16_t *W, int64_t M,
                      int64_t N, int64_t K, double *Y)
{
#pragma omp parallel for collapse(2) schedule(static) num_threads(g_threads) if (g_threads > 1)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(X[m * K + k]) * oracle_bf16_to_f64(W[n * K + k]);
            Y[m * N + n] = acc;
        }
    }
}
