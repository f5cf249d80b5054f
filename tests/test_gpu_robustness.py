"""Robustness of the CUDA path: outputs never spill past their buffers (guard
bands), and the bounded-wait failure path reports a timeout and leaves the
context usable -- exercised by a test-only injection that stops the
pipelines' producers, so the waits really run out, never by faulting the
GPU."""
import time

import numpy as np

import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu

GUARD = 64            # elements of canary on each side (128 bytes: keeps 16-byte alignment)
CANARY = 0x7FA5       # a BF16 NaN pattern no kernel writes


def _guarded(torch, n):
    buf = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.int16, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(torch.bfloat16)


def _check_guards(buf, n):
    h = host_bits16(buf)
    assert np.all(h[:GUARD] == CANARY) and np.all(h[GUARD + n:] == CANARY), "write outside the output"


@pytest.mark.parametrize("N,K", [(1, 128), (37, 384), (3000, 3840), (333, 15360)])
def test_gemv_writes_only_its_output(N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, seed=N + K)
    buf, y = _guarded(torch, N)
    w4.w4a16_gemv(dev_tensor(p["x"], torch.bfloat16).view(-1), dev_tensor(p["qw"], torch.uint8),
                  dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16), y)
    torch.cuda.synchronize()
    _check_guards(buf, N)
    assert_close(host_bits16(y), oracle.gemv_int4(p["x"], p["qw"], p["s"], p["z"], K=K), "guarded gemv")


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (130, 240, 384), (257, 464, 512)])
def test_gemm_writes_only_its_output(M, N, K):
    torch, w4 = cuda_or_skip()
    p = synth.int4_problem(N, K, M=M, seed=M * 7 + N)
    buf, y = _guarded(torch, M * N)
    w4.w4a16_gemm(dev_tensor(p["x"], torch.bfloat16).view(M, K), dev_tensor(p["qw"], torch.uint8),
                  dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16), y.view(M, N))
    torch.cuda.synchronize()
    _check_guards(buf, M * N)
    ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    assert_close(host_bits16(y).reshape(M, N), ref, "guarded gemm")


def test_moe_writes_only_its_output():
    torch, w4 = cuda_or_skip()
    E, N, K, topk = 5, 96, 448, 3
    m = synth.fp4_moe_problem(E, N, K, topk, seed=3)
    buf, y = _guarded(torch, topk * N)
    w4.fp4_moe_gemv(dev_tensor(m["x"], torch.bfloat16).view(-1), dev_tensor(m["qw"], torch.uint8),
                    dev_tensor(m["s"], torch.float16), dev_tensor(m["ids"], torch.int32), y.view(topk, N))
    torch.cuda.synchronize()
    _check_guards(buf, topk * N)
    ref, bad = oracle.moe_fp4(m["x"], m["qw"], m["s"], m["ids"], E=E, N=N, K=K)
    assert bad == 0
    assert_close(host_bits16(y).reshape(topk, N), ref, "guarded moe")


@pytest.mark.parametrize("flag", ["producers", "consumers"])
@pytest.mark.parametrize("kind", ["gemv", "moe", "gemm"])
def test_bounded_wait_reports_timeout_and_recovers(kind, flag):
    """flag "producers": no stage is ever issued, the consumers' waits run
    out.  flag "consumers": stages are issued but never taken, so the
    producers' waits for free stages run out with their copies issued; each
    producer then waits for its own copies before the launch ends."""
    torch, w4 = cuda_or_skip()
    assert w4.w4a16_check_device_error() == 0
    if kind == "gemv":
        p = synth.int4_problem(3000, 3840, seed=8)
        args = (dev_tensor(p["x"], torch.bfloat16).view(-1), dev_tensor(p["qw"], torch.uint8),
                dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16))
        run = lambda: w4.w4a16_gemv(*args)
        ref = oracle.gemv_int4(p["x"], p["qw"], p["s"], p["z"], K=3840)
    elif kind == "moe":
        E, N, K, topk = 8, 256, 1024, 3
        m = synth.fp4_moe_problem(E, N, K, topk, seed=4)
        args = (dev_tensor(m["x"], torch.bfloat16).view(-1), dev_tensor(m["qw"], torch.uint8),
                dev_tensor(m["s"], torch.float16), dev_tensor(m["ids"], torch.int32))
        run = lambda: w4.fp4_moe_gemv(*args)
        ref, _ = oracle.moe_fp4(m["x"], m["qw"], m["s"], m["ids"], E=E, N=N, K=K)
    else:
        M, N, K = 130, 448, 512
        p = synth.int4_problem(N, K, M=M, seed=9)
        args = (dev_tensor(p["x"], torch.bfloat16).view(M, K), dev_tensor(p["qw"], torch.uint8),
                dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16))
        run = lambda: w4.w4a16_gemm(*args)
        ref = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    w4.w4a16_debug_inject(w4.INJECT_STALL_PIPELINE if flag == "producers" else w4.INJECT_STALL_CONSUMERS)
    try:
        t0 = time.monotonic()
        run()
        status = w4.w4a16_check_device_error()  # synchronises; reads and clears
        waited = time.monotonic() - t0
    finally:
        w4.w4a16_debug_inject(0)
    assert status == 5  # W4A16_ERR_TIMEOUT
    # the waits ran out at their limit (about 2 s), not at once and not never
    assert 1.5 < waited < 30.0, waited
    # the context is usable and the same call is correct again
    y = run()
    torch.cuda.synchronize()
    assert w4.w4a16_check_device_error() == 0
    assert_close(host_bits16(y).reshape(ref.shape), ref, kind + " after recovery")


def test_pointers_must_be_memory_of_the_current_device():
    """A host pointer (here a 16-byte-aligned numpy buffer) passed as an
    activation is refused on the host with INVALID_ARG, and nothing runs."""
    import ctypes
    torch, w4 = cuda_or_skip()
    N, K = 64, 256
    p = synth.int4_problem(N, K, seed=2)
    qw, s, z = dev_tensor(p["qw"], torch.uint8), dev_tensor(p["s"], torch.float16), dev_tensor(p["z"], torch.float16)
    y = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    host = np.zeros(K + 8, dtype=np.uint16)
    off = (-host.ctypes.data % 16) // 2
    hx = host[off:off + K]
    assert hx.ctypes.data % 16 == 0
    lib = w4.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    r = lib.w4a16_gemv(ctypes.c_void_p(hx.ctypes.data), ctypes.c_void_p(qw.data_ptr()),
                       ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(z.data_ptr()),
                       ctypes.c_void_p(y.data_ptr()), N, K, 128, st)
    assert r == 1, r  # W4A16_ERR_INVALID_ARG
    assert "not device memory" in w4.w4a16_last_error_string() or "not CUDA memory" in w4.w4a16_last_error_string()
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(y.view(torch.int16))) == 0  # nothing was launched
    assert w4.w4a16_check_device_error() == 0
