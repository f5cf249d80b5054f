"""Prefill GEMM (tcgen05 tensor cores) through the C ABI vs the binary64 oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


def _run(w4, torch, p):
    Y = w4.w4a16_gemm(dev_tensor(p["x"], torch.bfloat16), dev_tensor(p["qw"], torch.uint8),
                      dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16))
    torch.cuda.synchronize()
    return host_bits16(Y).reshape(p["M"], p["N"])


# tails in M (not a multiple of 128) and N (not a multiple of 128), one
# K block pair (K = 128), several stages, the largest K
@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (3, 48, 256), (128, 128, 128), (130, 256, 512),
                                   (64, 1024, 3840), (257, 400, 384), (128, 16, 16384)])
def test_gemm_small_and_ragged(M, N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=M * 7 + N + K)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(_run(w4, torch, p), ref, "gemm %dx%dx%d" % (M, N, K))


# small batches on the tensor cores (M = 5..127: X tiles of M rounded up to
# 16 rows, one to eight 16-row blocks, the half of the accumulator past 64
# rows used or not) and N of any size: odd N with an odd group count, so the
# tile's scale and zero rows end inside a 16-byte chunk that must be
# zero-filled past the tensors' end
@pytest.mark.parametrize("M,N,K", [(5, 200, 256), (9, 113, 384), (16, 225, 640), (17, 150, 512),
                                   (31, 1001, 1920), (33, 7, 256), (48, 129, 768), (63, 337, 3840),
                                   (65, 96, 384), (80, 300, 640), (100, 113, 1024), (127, 64, 256),
                                   (130, 241, 384), (64, 15360, 3840)])
def test_gemm_small_m_and_any_n(M, N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=M * 13 + N + K)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(_run(w4, torch, p), ref, "gemm %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("M", [128, 2048])
def test_gemm_full_size_sampled(M):
    # M x 15360 x 3840 on the GPU; the oracle checks sampled rows and columns
    torch, w4 = cuda_or_skip()
    N, K = 15360, 3840
    p = synth.int4_problem(N, K, M=M, seed=0)
    Y = _run(w4, torch, p)
    rng = np.random.default_rng(M)
    cols = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N), rng.integers(0, N, 128)]))
    rows = np.unique(np.concatenate([np.arange(min(M, 32)), np.arange(M - 16, M), rng.integers(0, M, 16)]))
    ref = oracle.gemm_int4(p["x"][rows], p["qw"][cols], p["s"][cols], p["z"][cols], K=K)
    assert_close(Y[np.ix_(rows, cols)], ref, "gemm M=%d sample" % M)


def test_gemm_identity_weights():
    torch, w4 = cuda_or_skip()
    K = 256
    codes = np.eye(K, dtype=np.uint8)
    qw = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    one = np.float16(1.0).view(np.uint16)
    p = {"qw": qw, "s": np.full((K, 2), one, np.uint16), "z": np.zeros((K, 2), np.uint16),
         "x": synth.normal_bf16(synth.Stream(3), (200, K)), "M": 200, "N": K}
    # y = x up to the binary32 cancellation of the 128 * sum(x) offset
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    y = _run(w4, torch, p)
    assert_close(y, ref, "identity")
    assert np.mean(y == p["x"]) > 0.99


def test_gemm_repeatable():
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(512, 1024, M=256, seed=4)
    a = _run(w4, torch, p)
    b = _run(w4, torch, p)
    assert np.array_equal(a, b)
    assert w4.w4a16_check_device_error() == 0


def test_gemm_large_activations_keep_bf16_range():
    # X enters the tensor cores as loaded BF16: magnitudes far beyond the F16
    # range are fine
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(256, 512, M=8, seed=6)
    xb = (p["x"].astype(np.uint32) << 16).view(np.float32) * np.float32(1e6)
    p["x"] = torch.tensor(xb).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=512)
    assert_close(_run(w4, torch, p), ref, "gemm large x")
    assert w4.w4a16_check_device_error() == 0


def test_gemm_fractional_zero_points():
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(384, 1024, M=64, seed=8)
    rng = np.random.default_rng(8)
    p["z"] = rng.uniform(0, 15, size=p["z"].shape).astype(np.float16).view(np.uint16)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=1024)
    assert_close(_run(w4, torch, p), ref, "gemm fractional z")
