"""Activations with a wide range inside a 128-element group, through every
INT4 entry point, against the binary64 oracle at the product tolerance.

Each group of every activation row gets one value 2^10, 2^12 or 2^14 times
larger than the N(0, 1) rest.  In the "zeroed" variant the weight of that
column is exactly zero in every row (its code equals the integer zero point),
so every output is built from the small values alone: a kernel that rounds
the small activations against the group maximum shows it there."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, cuda_or_skip, dev_tensor, host_bits16


def _bf16_bits(v):
    return (np.asarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _outlier_problem(M, N, K, ratio_log2, zeroed, seed):
    """An INT4 problem whose activation rows hold one outlier per group at a
    seeded column shared by the rows (exact powers of two, random signs)."""
    p = synth.int4_problem(N, K, M=M, seed=seed)
    G = K // 128
    rng = np.random.default_rng(seed)
    cols = np.arange(G) * 128 + rng.integers(0, 128, G)
    X = p["x"].reshape(M, K).copy()
    signs = np.where(rng.integers(0, 2, (M, G)) == 0, -1.0, 1.0)
    X[:, cols] = _bf16_bits(signs * 2.0 ** ratio_log2)
    p["x"] = X
    if zeroed:
        qw = p["qw"].copy()
        zf = p["z"].view(np.float16).astype(np.float64)        # integer zero points 0..15
        for g, c in enumerate(cols):
            code = zf[:, g].astype(np.uint8)                   # q = z: the weight is exactly 0
            b = qw[:, c // 2]
            qw[:, c // 2] = np.where(c % 2 == 0, (b & 0xF0) | code, (b & 0x0F) | (code << 4))
        p["qw"] = qw
    return p


def _check(y_bits, p, M, N, K, what):
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(y_bits.reshape(M, N), ref, what)


@pytest.mark.gpu
@pytest.mark.parametrize("zeroed", [False, True])
@pytest.mark.parametrize("ratio_log2", [10, 12, 14])
@pytest.mark.parametrize("N,K", [(257, 3840), (96, 15360)])
def test_gemv_group_outliers(N, K, ratio_log2, zeroed):
    torch, w4 = cuda_or_skip()
    p = _outlier_problem(1, N, K, ratio_log2, zeroed, seed=ratio_log2 * 10 + zeroed)
    y = w4.w4a16_gemv(dev_tensor(p["x"], torch.bfloat16).view(-1), dev_tensor(p["qw"], torch.uint8),
                      dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16))
    torch.cuda.synchronize()
    _check(host_bits16(y), p, 1, N, K, "gemv outliers 2^%d%s" % (ratio_log2, " zeroed" if zeroed else ""))


@pytest.mark.gpu
@pytest.mark.parametrize("zeroed", [False, True])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 16, 130])
def test_gemm_group_outliers(M, zeroed):
    """M = 2..4 take the streaming pass, larger M the tensor cores."""
    torch, w4 = cuda_or_skip()
    N, K = 224, 3840
    p = _outlier_problem(M, N, K, 14, zeroed, seed=M * 3 + zeroed)
    Y = w4.w4a16_gemm(dev_tensor(p["x"], torch.bfloat16).view(M, K), dev_tensor(p["qw"], torch.uint8),
                      dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16))
    torch.cuda.synchronize()
    _check(host_bits16(Y), p, M, N, K, "gemm M=%d outliers 2^14%s" % (M, " zeroed" if zeroed else ""))


def test_zeroed_outlier_construction_is_exact():
    """The zeroed variant really removes the outlier's contribution: the
    oracle's result equals that of the same activations with the outliers
    set to zero."""
    p = _outlier_problem(2, 64, 1024, 14, True, seed=1)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=1024)
    X = (p["x"].astype(np.uint32) << 16).view(np.float32)
    X = np.where(np.abs(X) >= 2.0 ** 14, 0.0, X).astype(np.float32)
    ref0 = oracle.gemm_int4(_bf16_bits(X), p["qw"], p["s"], p["z"], K=1024)
    assert np.array_equal(ref, ref0)
