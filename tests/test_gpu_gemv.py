"""Decode GEMV (M = 1) through the C ABI vs the binary64 oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


def _run(w4, torch, p):
    K = p["K"]
    y = w4.w4a16_gemv(dev_tensor(p["x"], torch.bfloat16).view(-1),
                      dev_tensor(p["qw"], torch.uint8),
                      dev_tensor(p["s"], torch.float16),
                      dev_tensor(p["z"], torch.float16))
    torch.cuda.synchronize()
    return host_bits16(y)


# small and ragged shapes: odd N, odd group count (K = 384, 1920), one group,
# the largest supported K, several stages per CTA
@pytest.mark.parametrize("N,K", [(1, 128), (2, 128), (7, 384), (33, 1920), (1000, 3840),
                                 (333, 15360), (64, 16384), (4099, 256)])
def test_gemv_small_and_ragged(N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, seed=N * 31 + K)
    ref = oracle.gemv_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(_run(w4, torch, p), ref, "gemv %dx%d" % (N, K))


@pytest.mark.parametrize("N,K", [(3840, 3840), (15360, 3840), (3840, 15360)])
def test_gemv_full_size_configs(N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, seed=0)
    ref = oracle.gemv_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(_run(w4, torch, p), ref, "gemv %dx%d" % (N, K))


def test_gemv_vocab_sampled_rows():
    # 262144 x 3840: the whole product on the GPU, 3072 rows checked
    torch, w4 = cuda_or_skip()
    N, K = 262144, 3840
    p = synth.int4_problem(N, K, seed=0)
    y = _run(w4, torch, p)
    rows = np.unique(np.concatenate([np.arange(512), np.arange(N - 512, N),
                                     np.random.default_rng(0).integers(0, N, 2048)]))
    ref = oracle.gemv_int4(p["x"], p["qw"][rows], p["s"][rows], p["z"][rows], K=K)
    assert_close(y[rows], ref, "vocab sample")


@pytest.mark.parametrize("scale", [1e-20, 1e4])
def test_gemv_activation_scales(scale):
    torch, w4 = cuda_or_skip()
    N, K = 257, 3840
    p = synth.int4_problem(N, K, seed=5)
    x = (p["x"].astype(np.uint32) << 16).view(np.float32) * np.float32(scale)
    p["x"] = (x.view(np.uint32) >> 16).astype(np.uint16)  # exact: power-free scale ok
    p["x"] = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = oracle.gemv_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    y = _run(w4, torch, p)
    yv = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rel = np.linalg.norm(yv - ref) / np.linalg.norm(ref)
    assert rel <= 5e-3


def test_gemv_closed_forms():
    torch, w4 = cuda_or_skip()
    N, K = 100, 1024
    p = synth.int4_problem(N, K, seed=9)
    p["qw"][:] = 0
    p["z"][:] = np.float16(0).view(np.uint16)
    assert np.all(_run(w4, torch, p) == 0)                 # all-zero codes -> 0
    p["qw"][:] = 0xFF                                      # all-15 codes, constant s
    p["s"][:] = np.float16(3.0 / 256).view(np.uint16)
    ref = oracle.gemv_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(_run(w4, torch, p), ref, "all-15")


def test_gemv_deterministic_and_repeatable():
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(3000, 3840, seed=3)
    a = _run(w4, torch, p)
    b = _run(w4, torch, p)
    assert np.array_equal(a, b)
    assert w4.w4a16_check_device_error() == 0


def test_gemv_rejects_bad_arguments_without_launch():
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(16, 256, seed=1)
    x = dev_tensor(p["x"], torch.bfloat16).view(-1)
    qw = dev_tensor(p["qw"], torch.uint8)
    s64 = torch.zeros(16 * 4, dtype=torch.float16, device="cuda")
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemv(x, qw, s64, s64, group=64)
    assert e.value.status == 2
    big = torch.empty(16 * 8192 + 8, dtype=torch.uint8, device="cuda")
    mis = big[8:].view(16, 8192)                   # 8-byte aligned only
    with pytest.raises(w4.W4A16Error) as e:
        w4.w4a16_gemv(torch.zeros(16384, dtype=torch.bfloat16, device="cuda"), mis,
                      torch.zeros(16 * 128, dtype=torch.float16, device="cuda"),
                      torch.zeros(16 * 128, dtype=torch.float16, device="cuda"))
    assert e.value.status == 3


def test_gemv_stream_order_with_early_launch():
    """The GEMV may start before the previous kernel of the stream ends
    (programmatic dependent launch): it must still see an activation, weights
    and output buffer that the previous kernels wrote, with no host sync in
    between.  Chain: torch writes x, up GEMV, down GEMV on the up output,
    torch rewrites the weights and poisons y, GEMV again."""
    torch, w4 = cuda_or_skip()
    up = synth.int4_problem(15360, 3840, seed=21)
    dn = synth.int4_problem(3840, 15360, seed=22)
    qu, su, zu = (dev_tensor(up["qw"], torch.uint8), dev_tensor(up["s"], torch.float16),
                  dev_tensor(up["z"], torch.float16))
    qd, sd, zd = (dev_tensor(dn["qw"], torch.uint8), dev_tensor(dn["s"], torch.float16),
                  dev_tensor(dn["z"], torch.float16))
    x0 = dev_tensor(up["x"], torch.bfloat16).view(-1)
    torch.cuda.synchronize()
    x = x0 * 2.0                              # written by a kernel just before the GEMV
    y_up = w4.w4a16_gemv(x, qu, su, zu)
    y_dn = w4.w4a16_gemv(y_up, qd, sd, zd)    # consumes the previous launch's output
    qd2 = torch.flip(qd, dims=[0]).contiguous()  # weights written just before use
    y2 = torch.full((3840,), float("nan"), dtype=torch.bfloat16, device="cuda")
    w4.w4a16_gemv(y_up, qd2, sd, zd, y2)
    torch.cuda.synchronize()
    xh = host_bits16(x)
    ref_up = oracle.gemv_int4(xh, up["qw"], up["s"], up["z"], K=3840)
    yu = host_bits16(y_up)
    assert_close(yu, ref_up, "chained up")
    ref_dn = oracle.gemv_int4(yu, dn["qw"], dn["s"], dn["z"], K=15360)
    assert_close(host_bits16(y_dn), ref_dn, "chained down")
    ref_2 = oracle.gemv_int4(yu, dn["qw"][::-1].copy(), dn["s"], dn["z"], K=15360)
    assert_close(host_bits16(y2), ref_2, "rewritten weights")
    assert w4.w4a16_check_device_error() == 0
