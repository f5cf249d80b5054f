"""The binary16-operand prefill GEMM (w4a16_gemm_f16) through the C ABI vs
the binary64 oracle: the product tolerance on the synthetic workloads, and
the error bound its arithmetic gives (each weight rounded once to binary16)
on activations with outliers far above the rest."""
import time

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, bf16_to_f64, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


def _run(w4, torch, p, sym=False):
    z = None if sym else dev_tensor(p["z"], torch.float16)
    Y = w4.w4a16_gemm_f16(dev_tensor(p["x"], torch.bfloat16).view(p["M"], p["K"]), dev_tensor(p["qw"], torch.uint8),
                          dev_tensor(p["s"], torch.float16), z)
    torch.cuda.synchronize()
    return host_bits16(Y).reshape(p["M"], p["N"])


# one token tile and several (256 rows each), ragged M and N, one group and the largest K;
# K = 4096 / 4224 / 6144 / 16384: the pre-pass holding 2 (all used) / 3 of 4 / 3 of 4 / 8
# blocks of 8 values per thread
@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (9, 113, 384), (16, 225, 640), (64, 1024, 3840),
                                   (128, 128, 128), (130, 256, 512), (257, 400, 384), (300, 129, 1920),
                                   (513, 96, 768), (128, 16, 16384), (40, 130, 4096), (70, 200, 4224),
                                   (33, 300, 6144)])
def test_gemm_f16_small_and_ragged(M, N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=M * 5 + N + K)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(_run(w4, torch, p), ref, "gemm_f16 %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", [(20, 200, 512), (300, 136, 1024)])
def test_gemm_f16_symmetric(M, N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=M + N + K)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], None, K=K)
    assert_close(_run(w4, torch, p, sym=True), ref, "gemm_f16 symmetric")


# More tiles than SMs (several waves of CTAs), ragged in M and N, with one to
# several packed-code stages a tile and one to four issuers.  Every output
# column is checked on a sample of token rows (the oracle's cost grows with
# M x N x K).
@pytest.mark.parametrize("M,N,K,sym", [
    (600, 20100, 512, False),   # 3 token tiles (the last of 88 rows) x 158 weight tiles (the last of 4 rows)
    (600, 20100, 512, True),    # the same, symmetric
    (1000, 5000, 768, False),   # 4 x 40 tiles, three packed-code stages a tile
    (100, 20600, 1024, False),  # 112-row token tiles: two issuers, 161 tiles
    (40, 20000, 256, False),    # 48-row token tiles: four issuers, one packed-code stage a tile
    (600, 20100, 384, False),   # K % 256 == 128: a half packed-code stage ends every tile
    (256, 20096, 2048, False),  # 157 tiles: the 5 past the full wave split 4 ways along K
    (300, 10000, 1024, False),  # 158 tiles, ragged M and N: the 6 past the full wave split 2 ways
    (300, 10000, 1024, True),   # the same, symmetric
])
def test_gemm_f16_many_tiles(M, N, K, sym):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=M + N + K + sym)
    y = _run(w4, torch, p, sym=sym)
    rows = np.unique(np.array([0, 1, M // 2, M - 2, M - 1] + [r for r in (255, 256, 511, 512) if r < M]))
    ref = oracle.gemm_int4(p["x"].reshape(M, K)[rows], p["qw"], p["s"], None if sym else p["z"], K=K)
    assert_close(y[rows], ref, "gemm_f16 %dx%dx%d%s sampled" % (M, N, K, " symmetric" if sym else ""))


def test_gemm_f16_full_size_sampled():
    # the prefill shape: every output on the GPU, a sample of tokens on the oracle
    torch, w4 = cuda_or_skip()
    M, N, K = 2048, 15360, 3840
    p = synth.int4_problem(N, K, M=M, seed=3)
    y = _run(w4, torch, p)
    rows = np.array([0, 1, 255, 256, 1000, 2047])
    ref = oracle.gemm_int4(p["x"].reshape(M, K)[rows], p["qw"], p["s"], p["z"], K=K)
    assert_close(y[rows], ref, "gemm_f16 2048x15360x3840 sampled")


@pytest.mark.parametrize("ratio_log2", [10, 14])
@pytest.mark.parametrize("M", [16, 300])
def test_gemm_f16_outliers_within_the_bound(M, ratio_log2):
    """One activation per group 2^10 or 2^14 above the N(0, 1) rest: the
    error stays within the bound of one binary16 rounding per weight,
    2^-10 sum_k |x_k w_k| (twice the unit roundoff 2^-11, for the binary32
    sums), plus the BF16 rounding of the output (2^-8 |y|)."""
    torch, w4 = cuda_or_skip()
    N, K = 224, 3840
    p = synth.int4_problem(N, K, M=M, seed=M + ratio_log2)
    rng = np.random.default_rng(M + ratio_log2)
    G = K // 128
    cols = np.arange(G) * 128 + rng.integers(0, 128, G)
    X = p["x"].reshape(M, K).copy()
    signs = np.where(rng.integers(0, 2, (M, G)) == 0, -1.0, 1.0)
    X[:, cols] = (np.asarray(signs * 2.0 ** ratio_log2, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    p["x"] = X
    ref = oracle.gemm_int4(X, p["qw"], p["s"], p["z"], K=K)
    W = oracle.dequant_int4(p["qw"], p["s"], p["z"], K=K).astype(np.float64)
    bound = 2.0 ** -10 * (np.abs(bf16_to_f64(X)) @ np.abs(W).T) + 2.0 ** -8 * np.abs(ref) + 1e-30
    y = bf16_to_f64(_run(w4, torch, p))
    err = np.abs(y - ref)
    i = int(np.argmax(err / bound))
    assert np.all(err <= bound), "element %d: error %r, bound %r" % (i, err.flat[i], bound.flat[i])


def test_gemm_f16_bounded_wait_reports_timeout_and_recovers():
    """Stages issued but never taken: the producers' waits run out (K large
    enough that every ring wraps), the status reports the timeout and the
    next call is correct."""
    torch, w4 = cuda_or_skip()
    M, N, K = 130, 448, 2048
    p = synth.int4_problem(N, K, M=M, seed=9)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    for flag in (w4.INJECT_STALL_PIPELINE, w4.INJECT_STALL_CONSUMERS):
        assert w4.w4a16_check_device_error() == 0
        w4.w4a16_debug_inject(flag)
        try:
            t0 = time.monotonic()
            _run(w4, torch, p)
            status = w4.w4a16_check_device_error()
            waited = time.monotonic() - t0
        finally:
            w4.w4a16_debug_inject(0)
        assert status == 5  # W4A16_ERR_TIMEOUT
        assert 1.5 < waited < 30.0, waited
        assert_close(_run(w4, torch, p), ref, "gemm_f16 after recovery")
        assert w4.w4a16_check_device_error() == 0


def test_gemm_f16_many_tiles_bounded_wait_reports_timeout_and_recovers():
    """The same with more tiles than SMs: every CTA's waits run out, the
    status reports the timeout, each CTA leaves, and the next call is
    correct."""
    torch, w4 = cuda_or_skip()
    M, N, K = 300, 20100, 1024  # 2 x 158 tiles
    p = synth.int4_problem(N, K, M=M, seed=10)
    rows = np.array([0, 1, 150, 255, 256, 299])
    ref = oracle.gemm_int4(p["x"].reshape(M, K)[rows], p["qw"], p["s"], p["z"], K=K)
    for flag in (w4.INJECT_STALL_PIPELINE, w4.INJECT_STALL_CONSUMERS):
        assert w4.w4a16_check_device_error() == 0
        w4.w4a16_debug_inject(flag)
        try:
            t0 = time.monotonic()
            _run(w4, torch, p)
            status = w4.w4a16_check_device_error()
            waited = time.monotonic() - t0
        finally:
            w4.w4a16_debug_inject(0)
        assert status == 5  # W4A16_ERR_TIMEOUT
        assert 1.5 < waited < 30.0, waited
        assert_close(_run(w4, torch, p)[rows], ref, "gemm_f16 many tiles after recovery")
        assert w4.w4a16_check_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(300, 136, 512), (300, 10000, 1024)])
def test_gemm_f16_in_a_captured_graph(M, N, K):
    """The pre-pass scratch comes from a stream-ordered pool, so the call can
    be captured: replays after the inputs change give the new result (the
    second shape: 158 tiles, the 6 past the full wave split along K and
    finished by the reduction launch, all inside the graph)."""
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=21)
    X = dev_tensor(p["x"], torch.bfloat16).view(M, K)
    qw, s, z = dev_tensor(p["qw"], torch.uint8), dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        w4.w4a16_gemm_f16(X, qw, s, z, Y)  # warm-up outside capture
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            w4.w4a16_gemm_f16(X, qw, s, z, Y)
    for seed in (22, 23):
        q = synth.int4_problem(N, K, M=M, seed=seed)
        X.copy_(dev_tensor(q["x"], torch.bfloat16).view(M, K))
        g.replay()
        torch.cuda.synchronize()
        rows = np.array([0, 1, M // 2, M - 1])
        ref = oracle.gemm_int4(q["x"].reshape(M, K)[rows], p["qw"], p["s"], p["z"], K=K)
        assert_close(host_bits16(Y).reshape(M, N)[rows], ref, "gemm_f16 graph replay")
    assert w4.w4a16_check_device_error() == 0


@pytest.mark.parametrize("entry,M", [("w4a16_gemm_f16", 300), ("w4a16_gemm_f16", 16),
                                     ("w4a16_gemm", 300), ("w4a16_gemm", 16)])
def test_back_to_back_call_reads_the_previous_output(entry, M):
    """Two calls on one stream with no synchronisation between them, the
    second reading the first's output (consecutive launches may overlap by
    programmatic dependent launch and must still wait for what they read):
    each result matches the oracle on its actual input."""
    torch, w4 = cuda_or_skip()
    fn = getattr(w4, entry)
    K1, N1, N2 = 256, 384, 256
    p1 = synth.int4_problem(N1, K1, M=M, seed=31 + M)
    p2 = synth.int4_problem(N2, N1, M=M, seed=32 + M)
    X = dev_tensor(p1["x"], torch.bfloat16).view(M, K1)
    w1 = (dev_tensor(p1["qw"], torch.uint8), dev_tensor(p1["s"], torch.float16), dev_tensor(p1["z"], torch.float16))
    w2 = (dev_tensor(p2["qw"], torch.uint8), dev_tensor(p2["s"], torch.float16), dev_tensor(p2["z"], torch.float16))
    Y1 = torch.empty(M, N1, dtype=torch.bfloat16, device="cuda")
    Y2 = torch.empty(M, N2, dtype=torch.bfloat16, device="cuda")
    for _ in range(3):  # each round's first call overwrites what the previous second call read
        fn(X, *w1, Y1)
        fn(Y1, *w2, Y2)
    torch.cuda.synchronize()
    y1 = host_bits16(Y1).reshape(M, N1)
    y2 = host_bits16(Y2).reshape(M, N2)
    assert_close(y1, oracle.gemm_int4(p1["x"], p1["qw"], p1["s"], p1["z"], K=K1), "%s first call" % entry)
    assert_close(y2, oracle.gemm_int4(y1.reshape(-1), p2["qw"], p2["s"], p2["z"], K=N1), "%s second call" % entry)
    assert w4.w4a16_check_device_error() == 0
