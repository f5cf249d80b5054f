"""w4a16_copy: the kernel copy for a decode step's small transfers (device
memory and pinned, mapped host memory) -- byte-exact, any size and alignment,
ordered with the library's launches, capturable in a CUDA graph."""
import ctypes

import numpy as np
import pytest

import synth
from tests.gpu_helpers import cuda_or_skip, dev_tensor

pytestmark = pytest.mark.gpu

SIZES = [0, 1, 15, 16, 17, 4095, 38400, (1 << 20) + 3]


def _bytes(torch, n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("kind", ["d2d", "h2d", "d2h", "h2h"])
def test_copy_bytes_exact(kind, n):
    torch, w4 = cuda_or_skip()
    src_h = _bytes(torch, n, n + 1)
    src = src_h.cuda() if kind[0] == "d" else src_h.pin_memory()
    dst = torch.full((n,), 0xA5, dtype=torch.uint8)
    dst = dst.cuda() if kind[2] == "d" else dst.pin_memory()
    w4.w4a16_copy(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src_h)


@pytest.mark.parametrize("off_d,off_s", [(1, 0), (0, 3), (5, 7), (8, 8)])
def test_copy_misaligned_ends(off_d, off_s):
    # byte offsets: the kernel falls back to byte moves unless both ends are 16-aligned
    torch, w4 = cuda_or_skip()
    n = 1000
    src_h = _bytes(torch, n + 16, 7)
    src = src_h.pin_memory()
    dst = torch.zeros(n + 16, dtype=torch.uint8, device="cuda")
    w4.w4a16_copy(dst[off_d:off_d + n], src[off_s:off_s + n])
    torch.cuda.synchronize()
    out = dst.cpu()
    assert torch.equal(out[off_d:off_d + n], src_h[off_s:off_s + n])
    assert int(out[:off_d].sum()) == 0 and int(out[off_d + n:].sum()) == 0  # nothing written outside


def test_copy_refuses_pageable_host_memory_before_launch():
    # through the C ABI directly: a pageable numpy buffer is refused on the host
    torch, w4 = cuda_or_skip()
    lib = w4.lib()
    host = np.zeros(64, np.uint8)
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    r = lib.w4a16_copy(ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(host.ctypes.data), 64, st)
    assert r == 1
    assert b"cannot reach" in lib.w4a16_last_error_string()
    r = lib.w4a16_copy(ctypes.c_void_p(host.ctypes.data), ctypes.c_void_p(dev.data_ptr()), 64, st)
    assert r == 1
    torch.cuda.synchronize()
    assert w4.w4a16_check_device_error() == 0


def test_copy_gemv_copy_in_a_graph():
    # a decode step as the benchmark's end-to-end run makes it: pinned x in,
    # the GEMV, y out to pinned memory, captured once and replayed with new x
    torch, w4 = cuda_or_skip()
    N, K = 1000, 3840
    p = synth.int4_problem(N, K, seed=5)
    qw, s, z = (dev_tensor(p["qw"], torch.uint8), dev_tensor(p["s"], torch.float16),
                dev_tensor(p["z"], torch.float16))
    x_pin = torch.empty(K, dtype=torch.bfloat16).pin_memory()
    y_pin = torch.empty(N, dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty(K, dtype=torch.bfloat16, device="cuda")
    y_d = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    x_pin.copy_(dev_tensor(p["x"], torch.bfloat16).reshape(-1).cpu())
    w4.w4a16_copy(x_d, x_pin)  # first calls (the library's per-device set-up) outside the capture
    w4.w4a16_gemv(x_d, qw, s, z, y_d)
    w4.w4a16_copy(y_pin, y_d)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.w4a16_copy(x_d, x_pin)
        w4.w4a16_gemv(x_d, qw, s, z, y_d)
        w4.w4a16_copy(y_pin, y_d)
    for seed in (11, 12):
        xs = synth.int4_problem(N, K, seed=seed)["x"]
        x_pin.copy_(dev_tensor(xs, torch.bfloat16).reshape(-1).cpu())
        g.replay()
        torch.cuda.synchronize()
        ref = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        w4.w4a16_gemv(dev_tensor(xs, torch.bfloat16).reshape(-1), qw, s, z, ref)
        torch.cuda.synchronize()
        assert torch.equal(y_pin.view(torch.int16), ref.cpu().view(torch.int16))
    assert w4.w4a16_check_device_error() == 0
