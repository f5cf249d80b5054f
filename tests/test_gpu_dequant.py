"""Debug dequant entry vs the oracle: bit-exact (binary32 and bfloat16)."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


def _int4_case(N, K, seed, z_fractional=False):
    p = synth.int4_problem(N, K, seed=seed)
    if z_fractional:  # arbitrary FP16 zero points, negative scales included
        rng = np.random.default_rng(seed)
        p["z"] = rng.uniform(-3, 18, size=p["z"].shape).astype(np.float16).view(np.uint16)
        p["s"] = rng.uniform(-0.05, 0.05, size=p["s"].shape).astype(np.float16).view(np.uint16)
    return p


@pytest.mark.parametrize("N,K,frac", [(1, 128, False), (37, 384, True), (300, 3840, False),
                                      (5, 16384, True), (3840, 3840, False)])
def test_int4_dequant_bit_exact(N, K, frac):
    torch, w4 = cuda_or_skip()
    p = _int4_case(N, K, seed=N + K, z_fractional=frac)
    qw, s, z = (dev_tensor(p["qw"], torch.uint8), dev_tensor(p["s"], torch.float16),
                dev_tensor(p["z"], torch.float16))
    ref = oracle.dequant_int4(p["qw"], p["s"], p["z"], K=K)
    out32 = w4.w4a16_dequant(w4.FMT_INT4, qw, s, z, out_dtype=w4.OUT_F32)
    got = out32.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    out16 = w4.w4a16_dequant(w4.FMT_INT4, qw, s, z, out_dtype=w4.OUT_BF16)
    assert np.array_equal(host_bits16(out16).reshape(N, K),
                          oracle.round_bf16(ref.astype(np.float64)).reshape(N, K))


def test_int4_dequant_vocab_rows_sampled():
    # full-size vocab matrix on the device; a contiguous row window checked
    torch, w4 = cuda_or_skip()
    N, K = 262144, 3840
    p = synth.int4_problem(N, K, seed=0)
    lo, hi = N - 1000, N
    ref = oracle.dequant_int4(p["qw"][lo:hi], p["s"][lo:hi], p["z"][lo:hi], K=K)
    qw = dev_tensor(p["qw"], torch.uint8)
    s = dev_tensor(p["s"], torch.float16)
    z = dev_tensor(p["z"], torch.float16)
    out = w4.w4a16_dequant(w4.FMT_INT4, qw[lo:hi], s[lo:hi], z[lo:hi], out_dtype=w4.OUT_F32)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("rows,K", [(1, 32), (7, 96), (64, 7168)])
def test_fp4_dequant_bit_exact(rows, K):
    torch, w4 = cuda_or_skip()
    st = synth.Stream(rows * 7 + K)
    qw = synth.packed_codes(st, rows, K)
    s = synth.uniform_f16(st, (rows, K // 32), -0.1, 0.1)
    ref = oracle.dequant_fp4(qw, s, K=K)
    dq, ds = dev_tensor(qw, torch.uint8), dev_tensor(s, torch.float16)
    out32 = w4.w4a16_dequant(w4.FMT_FP4, dq, ds, out_dtype=w4.OUT_F32)
    assert np.array_equal(out32.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    out16 = w4.w4a16_dequant(w4.FMT_FP4, dq, ds, out_dtype=w4.OUT_BF16)
    assert np.array_equal(host_bits16(out16).reshape(rows, K),
                          oracle.round_bf16(ref.astype(np.float64)))


def test_fp4_dequant_every_code():
    torch, w4 = cuda_or_skip()
    codes = np.arange(32) % 16
    qw = ((codes[1::2] << 4) | codes[0::2]).astype(np.uint8).reshape(1, 16)
    s = np.array([[np.float16(1.0).view(np.uint16)]], np.uint16)
    ref = oracle.dequant_fp4(qw, s, K=32)
    out = w4.w4a16_dequant(w4.FMT_FP4, dev_tensor(qw, torch.uint8), dev_tensor(s, torch.float16))
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
