"""Symmetric INT4 (no zero points: the code midpoint 8 for every group, the
symmetric GPTQ variant of "Lab 5", section "Quantisation correctness")
through every INT4 entry point, against the binary64 oracle with z = None."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


def _dev(torch, p):
    return (dev_tensor(p["qw"], torch.uint8), dev_tensor(p["s"], torch.float16))


@pytest.mark.parametrize("N,K", [(1, 128), (37, 384), (1000, 3840), (333, 15360), (15360, 3840)])
def test_gemv_symmetric(N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, seed=N * 7 + K + 1)
    qw, s = _dev(torch, p)
    y = w4.w4a16_gemv(dev_tensor(p["x"], torch.bfloat16).view(-1), qw, s, None)
    torch.cuda.synchronize()
    ref = oracle.gemv_int4(p["x"], p["qw"], p["s"], None, K=K)
    assert_close(host_bits16(y), ref, "symmetric gemv %dx%d" % (N, K))


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (130, 448, 512), (128, 1024, 3840), (257, 400, 384)])
def test_gemm_symmetric(M, N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=M + N + K)
    qw, s = _dev(torch, p)
    Y = w4.w4a16_gemm(dev_tensor(p["x"], torch.bfloat16).view(M, K), qw, s, None)
    torch.cuda.synchronize()
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], None, K=K)
    assert_close(host_bits16(Y).reshape(M, N), ref, "symmetric gemm %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("N,K", [(1, 128), (37, 384), (300, 3840)])
def test_dequant_symmetric_bit_exact(N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, seed=N + 2 * K)
    qw, s = _dev(torch, p)
    ref = oracle.dequant_int4(p["qw"], p["s"], None, K=K)
    got = w4.w4a16_dequant(w4.FMT_INT4, qw, s, None, out_dtype=w4.OUT_F32).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    out16 = w4.w4a16_dequant(w4.FMT_INT4, qw, s, None, out_dtype=w4.OUT_BF16)
    assert np.array_equal(host_bits16(out16).reshape(N, K),
                          oracle.round_bf16(ref.astype(np.float64)).reshape(N, K))


def test_symmetric_midpoint_codes_give_exact_zero():
    # every code 8: W = 0 exactly, so both paths must return +-0 bit patterns
    torch, w4 = cuda_or_skip()
    M, N, K = 3, 64, 384
    p = synth.int4_problem(N, K, M=M, seed=11)
    qw = torch.full((N, K // 2), 0x88, dtype=torch.uint8, device="cuda")
    s = dev_tensor(p["s"], torch.float16)
    X = dev_tensor(p["x"], torch.bfloat16).view(M, K)
    y = w4.w4a16_gemv(X[0].contiguous(), qw, s, None)
    Y = w4.w4a16_gemm(X, qw, s, None)
    torch.cuda.synchronize()
    assert np.all((host_bits16(y) & 0x7FFF) == 0)
    assert np.all((host_bits16(Y) & 0x7FFF) == 0)
