"""The unfused two-pass path ("Lab 5", section "Triton dequant + cuBLAS"):
w4a16_dequant writes BF16 weights, w4a16_bf16_gemm multiplies them (the
fusion ablation).  The dense GEMM is checked against the binary64 product of
the same BF16 operands; the two-pass result against its own definition and,
by the pages' relative RMSE, against the exact fused oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, bf16_to_f64, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(1, 16, 64), (130, 200, 256), (257, 384, 448), (128, 1024, 3840)])
def test_bf16_gemm_matches_binary64_product(M, N, K):
    torch, w4 = cuda_or_skip()
    X = synth.normal_bf16(synth.Stream(M * 3 + K), (M, K))
    W = synth.normal_bf16(synth.Stream(N * 5 + K), (N, K))
    Y = w4.w4a16_bf16_gemm(dev_tensor(X, torch.bfloat16).view(M, K), dev_tensor(W, torch.bfloat16).view(N, K))
    torch.cuda.synchronize()
    ref = oracle.gemm_bf16(X, W, K=K)
    assert_close(host_bits16(Y).reshape(M, N), ref, "bf16 gemm %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", [(3, 112, 256), (128, 448, 3840)])
def test_two_pass_int4(M, N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=N + K)
    qw, s, z = (dev_tensor(p["qw"], torch.uint8), dev_tensor(p["s"], torch.float16),
                dev_tensor(p["z"], torch.float16))
    Wb = w4.w4a16_dequant(w4.FMT_INT4, qw, s, z, out_dtype=w4.OUT_BF16)
    Y = w4.w4a16_bf16_gemm(dev_tensor(p["x"], torch.bfloat16).view(M, K), Wb)
    torch.cuda.synchronize()
    got = host_bits16(Y).reshape(M, N)
    # its own definition: BF16-rounded dequantised weights, exact product
    Wref = oracle.round_bf16(oracle.dequant_int4(p["qw"], p["s"], p["z"], K=K).astype(np.float64)).reshape(N, K)
    assert_close(got, oracle.gemm_bf16(p["x"], Wref, K=K), "two-pass %dx%dx%d" % (M, N, K))
    # against the exact fused result: the pages' relative RMSE criterion
    fused = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    rel = np.linalg.norm(bf16_to_f64(got) - fused) / np.linalg.norm(fused)
    assert rel <= 5e-3, rel


def test_bf16_gemm_full_size_sampled_columns():
    # M = 128 x N = 15360 x K = 3840 on the device; 64 output columns checked
    torch, w4 = cuda_or_skip()
    M, N, K = 128, 15360, 3840
    X = synth.normal_bf16(synth.Stream(41), (M, K))
    W = synth.normal_bf16(synth.Stream(42), (N, K))
    Y = w4.w4a16_bf16_gemm(dev_tensor(X, torch.bfloat16).view(M, K), dev_tensor(W, torch.bfloat16).view(N, K))
    torch.cuda.synchronize()
    cols = np.r_[0:16, 7000:7016, 15296:15312, 15344:15360]
    ref = oracle.gemm_bf16(X, W.reshape(N, K)[cols], K=K)
    assert_close(host_bits16(Y).reshape(M, N)[:, cols], ref, "bf16 gemm full-size columns")
