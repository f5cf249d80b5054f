"""The C ABI library: builds for sm_103a, loads, exports every declared
symbol, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT


@pytest.fixture(scope="module")
def libw4():
    from gemm_w4a16_gemv_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            names += re.findall(r"^(?:int64_t|int|const char \*)\s*(\w+)\s*\(", text, re.M)
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("w4a16_gemv", "w4a16_gemm", "w4a16_gemm_f16", "fp4_moe_gemv", "w4a16_dequant", "w4a16_bf16_gemm",
              "w4a16_check_device_error", "w4a16_last_error_string", "w4a16_version",
              "w4a16_debug_inject", "w4a16_linear_sequence", "w4a16_graph_create",
              "w4a16_graph_launch", "w4a16_graph_destroy", "w4a16_linear_chain",
              "w4a16_linear_chain_scratch_bytes", "w4a16_linear_chain_noalloc", "fp4_moe_gemm",
              "fp4_moe_gemm_scratch_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(libw4):
    import gemm_w4a16_gemv_gb300 as w4
    for n in declared_functions():
        assert hasattr(libw4, n), n
        assert n in w4.SIGNATURES, "binding lacks " + n


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import gemm_w4a16_gemv_gb300 as w4
    monkeypatch.setattr(w4, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(w4, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        w4.lib()


def _call(lib, name, *args):
    import gemm_w4a16_gemv_gb300 as w4
    fn = getattr(lib, name)
    fn.argtypes, fn.restype = w4.SIGNATURES[name]
    return fn(*args)


def test_host_validation_codes(libw4):
    # every case fails before any CUDA call, so it runs without a GPU
    A = 1 << 20      # a 16-byte aligned fake address; never dereferenced
    assert _call(libw4, "w4a16_gemv", None, A, A, A, A, 16, 256, 128, None) == 1
    assert _call(libw4, "w4a16_gemv", A, A, A, A, A, 0, 256, 128, None) == 1
    assert _call(libw4, "w4a16_gemv", A, A, A, A, A, 16, 256, 64, None) == 2
    assert _call(libw4, "w4a16_gemv", A, A, A, A, A, 16, 320, 128, None) == 1
    assert _call(libw4, "w4a16_gemv", A, A, A, A, A, 16, 32768, 128, None) == 2
    assert _call(libw4, "w4a16_gemv", A + 8, A, A, A, A, 16, 256, 128, None) == 3
    assert _call(libw4, "w4a16_gemm", A, A, A, A, A, 4, 24, 32768, 128, None) == 2  # K beyond 16384
    assert _call(libw4, "w4a16_gemm_f16", A, A, A, A, A, 4, 24, 32768, 128, None) == 2
    assert _call(libw4, "w4a16_gemm_f16", A, A, A, A, A, 4, 24, 3840, 64, None) == 2  # group
    assert _call(libw4, "w4a16_gemm_f16", A + 8, A, A, A, A, 4, 24, 3840, 128, None) == 3
    assert _call(libw4, "fp4_moe_gemv", A, A, A, A, 0, A, 4, 8, 128, 32, None) == 1
    assert _call(libw4, "fp4_moe_gemv", A, A, A, A, 2, A, 4, 8, 96, 32, None) == 1
    assert _call(libw4, "fp4_moe_gemv", A, A, A, A + 2, 2, A, 4, 8, 128, 32, None) == 3
    need = _call(libw4, "fp4_moe_gemm_scratch_bytes", 4, 2, 8, 512)
    assert need > 4 * 2 * 512 * 2 and need % 256 == 0
    assert _call(libw4, "fp4_moe_gemm_scratch_bytes", 0, 2, 8, 512) == 0
    assert _call(libw4, "fp4_moe_gemm_scratch_bytes", 8, 2, 8, 512) > need
    moe = lambda X, ids, M, K, g, scr, nb: _call(libw4, "fp4_moe_gemm", X, A, A, ids, M, 2, A, 8, 64, K, g,
                                                   scr, nb, None)
    assert moe(None, A, 4, 512, 32, A, need) == 1
    assert moe(A, A, 0, 512, 32, A, need) == 1
    assert moe(A, A, 4, 512, 16, A, need) == 2          # group other than 32
    assert moe(A, A, 4, 384, 32, A, need) == 2          # K not a multiple of 256
    assert moe(A + 8, A, 4, 512, 32, A, need) == 3
    assert moe(A, A + 2, 4, 512, 32, A, need) == 3      # ids not 4-byte aligned
    assert moe(A, A, 4, 512, 32, A + 16, need) == 3     # scratch not 256-byte aligned
    assert moe(A, A, 4, 512, 32, A, need - 1) == 1      # scratch too small
    assert _call(libw4, "w4a16_dequant", 1, A, A, A, A, 0, 4, 128, 32, None) == 1
    assert _call(libw4, "w4a16_dequant", 0, A, A, A, A, 2, 4, 128, 128, None) == 1
    assert _call(libw4, "w4a16_dequant", 0, A, A, A, A, 0, 4, 128, 64, None) == 2
    assert _call(libw4, "w4a16_bf16_gemm", None, A, A, 4, 16, 128, None) == 1
    assert _call(libw4, "w4a16_bf16_gemm", A, A, A, 4, 16, 96, None) == 1
    assert _call(libw4, "w4a16_bf16_gemm", A, A + 4, A, 4, 16, 128, None) == 3
    assert _call(libw4, "w4a16_dequant", 0, A, A, A, A, 0, 4, 128, 64, None) == 2
    msg = _call(libw4, "w4a16_last_error_string").decode()
    assert "group" in msg


def test_linear_struct_layout_matches_the_header():
    # five pointers then three int64: 64 bytes, no padding
    import gemm_w4a16_gemv_gb300 as w4
    assert ctypes.sizeof(w4.w4a16_linear) == 64
    assert w4.w4a16_linear.M.offset == 40 and w4.w4a16_linear.K.offset == 56


def test_sequence_and_graph_host_validation(libw4):
    # every case fails (or succeeds with nothing to do) before any CUDA call
    import gemm_w4a16_gemv_gb300 as w4
    A = 1 << 20
    ops = (w4.w4a16_linear * 3)()
    for i, (M, N, K) in enumerate([(1, 24, 256), (3, 32, 256), (1, 16, 384)]):
        ops[i].x = ops[i].qw = ops[i].s = ops[i].z = ops[i].y = A
        ops[i].M, ops[i].N, ops[i].K = M, N, K
    ops[2].K = 320                      # not a multiple of the group
    assert _call(libw4, "w4a16_linear_sequence", ops, 3, 128, None) == 1
    assert "op 2" in _call(libw4, "w4a16_last_error_string").decode()
    ops[2].K = 384
    ops[1].K = 32768                    # M > 1: the GEMM's rules, K <= 16384
    assert _call(libw4, "w4a16_linear_sequence", ops, 3, 128, None) == 2
    assert "op 1" in _call(libw4, "w4a16_last_error_string").decode()
    ops[1].K = 256
    ops[1].y = A + 8
    assert _call(libw4, "w4a16_linear_sequence", ops, 3, 128, None) == 3
    ops[1].y = A
    assert _call(libw4, "w4a16_linear_sequence", ops, 3, 64, None) == 2
    assert _call(libw4, "w4a16_linear_sequence", ops, -1, 128, None) == 1
    assert _call(libw4, "w4a16_linear_sequence", None, 2, 128, None) == 1
    assert _call(libw4, "w4a16_linear_sequence", None, 0, 128, None) == 0   # empty: nothing to launch
    h = ctypes.c_void_p(123)
    assert _call(libw4, "w4a16_graph_create", ops, 0, 128, ctypes.byref(h)) == 1
    assert h.value is None              # the handle is cleared on failure
    ops[0].qw = 0
    assert _call(libw4, "w4a16_graph_create", ops, 3, 128, ctypes.byref(h)) == 1
    assert "op 0" in _call(libw4, "w4a16_last_error_string").decode()
    assert _call(libw4, "w4a16_graph_create", ops, 3, 128, None) == 1
    assert _call(libw4, "w4a16_graph_launch", None, None) == 1
    assert _call(libw4, "w4a16_graph_destroy", None) == 0


def test_binding_checks_prebuilt_op_arrays():
    # a prebuilt array is never read past its length (checked before the call)
    import gemm_w4a16_gemv_gb300 as w4
    arr = (w4.w4a16_linear * 2)()
    with pytest.raises(ValueError, match="outside"):
        w4.w4a16_linear_sequence(arr, count=3)
    with pytest.raises(ValueError, match="outside"):
        w4.w4a16_linear_sequence(arr, count=-1)
    with pytest.raises(TypeError):
        w4.w4a16_linear_sequence((ctypes.c_int64 * 8)(), count=1)


def test_chain_host_validation(libw4):
    # every case fails (or has nothing to do) before any CUDA call
    import gemm_w4a16_gemv_gb300 as w4
    A = 1 << 20
    assert _call(libw4, "w4a16_linear_chain_scratch_bytes", 0) == 0
    assert _call(libw4, "w4a16_linear_chain_scratch_bytes", 2) == 12           # 2 counters + exit
    assert _call(libw4, "w4a16_linear_chain_scratch_bytes", 192) == 4 * 193
    assert _call(libw4, "w4a16_linear_chain_scratch_bytes", 193) == 4 * (193 + 2)  # two launches
    ops = (w4.w4a16_linear * 2)()
    base = [(A, A + 0x100000, A + 0x200000, A + 0x300000, A + 0x400000),
            (A + 0x500000, A + 0x600000, A + 0x700000, A + 0x800000, A + 0x900000)]
    for i in range(2):
        ops[i].x, ops[i].qw, ops[i].s, ops[i].z, ops[i].y = base[i]
        ops[i].M, ops[i].N, ops[i].K = 1, 64, 256
    S = A + 0xA00000
    assert _call(libw4, "w4a16_linear_chain", ops, 0, 128, None, 0, None) == 0  # nothing to launch
    assert _call(libw4, "w4a16_linear_chain", ops, 2, 128, None, 64, None) == 1  # null scratch
    assert _call(libw4, "w4a16_linear_chain", ops, 2, 128, S, 8, None) == 1      # too small
    assert "needed" in _call(libw4, "w4a16_last_error_string").decode()
    assert _call(libw4, "w4a16_linear_chain", ops, 2, 128, S + 2, 64, None) == 3  # misaligned
    ops[1].M = 2
    assert _call(libw4, "w4a16_linear_chain", ops, 2, 128, S, 64, None) == 2      # M = 1 only
    assert "op 1" in _call(libw4, "w4a16_last_error_string").decode()
    ops[1].M = 1
    ops[1].y = ops[1].x + 64                                                      # y inside its own x
    assert _call(libw4, "w4a16_linear_chain", ops, 2, 128, S, 64, None) == 1
    assert "own input" in _call(libw4, "w4a16_last_error_string").decode()
    ops[1].y = base[0][1] + 256                                                   # y inside op 0's codes
    assert _call(libw4, "w4a16_linear_chain", ops, 2, 128, S, 64, None) == 1
    assert "weights of op 0" in _call(libw4, "w4a16_last_error_string").decode()
    ops[1].y = S                                                                  # y on the scratch
    assert _call(libw4, "w4a16_linear_chain", ops, 2, 128, S, 64, None) == 1
    ops[1].y = base[1][4]
    ops[0].K = 320
    assert _call(libw4, "w4a16_linear_chain", ops, 2, 128, S, 64, None) == 1      # the GEMV's checks


def test_chain_noalloc_host_validation(libw4):
    # every case fails (or has nothing to do) before any CUDA call
    import gemm_w4a16_gemv_gb300 as w4
    A = 1 << 20
    ops = (w4.w4a16_linear * 4033)()
    for i in range(4033):
        ops[i].x, ops[i].qw, ops[i].s, ops[i].z, ops[i].y = A, A, A, A, A
        ops[i].M, ops[i].N, ops[i].K = 1, 16, 128
    assert _call(libw4, "w4a16_linear_chain_noalloc", ops, 0, 128, None) == 0    # nothing to do
    assert _call(libw4, "w4a16_linear_chain_noalloc", ops, 4033, 128, None) == 2  # beyond the built-in limit
    assert "4032" in _call(libw4, "w4a16_last_error_string").decode()
    ops[3].K = 320
    assert _call(libw4, "w4a16_linear_chain_noalloc", ops, 8, 128, None) == 1     # the GEMV's checks


def test_copy_host_validation(libw4):
    # null pointers and a negative size fail before any CUDA call
    A = 1 << 20
    assert _call(libw4, "w4a16_copy", None, A, 16, None) == 1
    assert _call(libw4, "w4a16_copy", A, None, 16, None) == 1
    assert _call(libw4, "w4a16_copy", A, A + 64, -1, None) == 1
    assert "bytes" in _call(libw4, "w4a16_last_error_string").decode()
    assert _call(libw4, "w4a16_copy", None, None, 0, None) == 0   # empty: nothing to launch


def test_copy_binding_refuses_pageable_host_tensors():
    # the binding refuses a host tensor that is not pinned before calling the library
    import torch
    import gemm_w4a16_gemv_gb300 as w4
    a, b = torch.zeros(8), torch.zeros(8)
    with pytest.raises(ValueError, match="pinned"):
        w4.w4a16_copy(a, b)
