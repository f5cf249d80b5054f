"""Decode-sized batches (M = 1..8) through w4a16_gemm: up to four rows share
one streaming pass over the weights (the M = 1 GEMV pipeline with one team set
per activation row), M = 5..8 run on the tensor cores with 16-row X tiles;
checked against the binary64 oracle."""
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


def _gemm(w4, torch, p, M, N, K, sym=False):
    Y = w4.w4a16_gemm(dev_tensor(p["x"], torch.bfloat16).view(M, K), dev_tensor(p["qw"], torch.uint8),
                      dev_tensor(p["s"], torch.float16), None if sym else dev_tensor(p["z"], torch.float16))
    torch.cuda.synchronize()
    return host_bits16(Y).reshape(M, N)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(16, 128), (112, 384), (1008, 3840), (336, 15360), (64, 16384)])
def test_small_batch_decode(M, N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=M * 1000 + N + K)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(_gemm(w4, torch, p, M, N, K), ref, "batched decode M=%d %dx%d" % (M, N, K))


@pytest.mark.parametrize("M", [2, 4, 6, 8])
def test_small_batch_decode_full_width(M):
    torch, w4 = cuda_or_skip()
    N, K = 15360, 3840
    p = synth.int4_problem(N, K, M=M, seed=77 + M)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(_gemm(w4, torch, p, M, N, K), ref, "batched decode M=%d full width" % M)


@pytest.mark.parametrize("M", [2, 3, 5, 7])
def test_small_batch_decode_symmetric(M):
    torch, w4 = cuda_or_skip()
    N, K = 496, 1920
    p = synth.int4_problem(N, K, M=M, seed=5 + M)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], None, K=K)
    assert_close(_gemm(w4, torch, p, M, N, K, sym=True), ref, "symmetric batched decode M=%d" % M)
