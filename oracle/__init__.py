"""CPU oracle for the fused W4A16 / FP4 products — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes it, and the two share no
code: this package compiles ``w4a16_oracle.c`` on its own with the host C
compiler and calls it through ctypes.

What it computes (page titles as published):
  * "Lab 5: Gemma4 end-to-end inference optimisation", sections "Quantisation
    correctness" and "Final configuration" (INT4, group 128, asymmetric, FP16
    scale) and "INT4 fused GEMV" (unpack, per-group scale/zero, dot product);
  * "DeepSeek V4 Triton FP4 optimisation in practice", deep analysis item 2
    (even K column <-> low nibble) and the FP4 expert GEMMs;
  * the problem statement y = x W^T, W = (q - z) * s, FP16 s and z;
  * symmetric INT4 (the symmetric GPTQ variant of "Quantisation correctness")
    in GPTQ's form: z = None means the implicit zero point 8;
  * the OCP MX definition of E2M1 for the FP4 value table;
  * the dense BF16 product of the unfused two-pass path ("Triton dequant +
    cuBLAS"), for the fusion ablation;
  * the batched-expert FP4 GEMM for M tokens routed to topk experts each (the
    pages' FP4 expert GEMMs at M > 1).

Every function here is pinned by ``tests/test_oracle_pins.py`` against
hand-written fixtures, closed forms, brute force and library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no FP contraction); return the path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-Wall", "-shared",
           "-fPIC", _SRC, "-o", tmp, "-lm"]
    # OpenMP only spreads independent output elements over threads (for the
    # timed all-cores baseline); without it the same code runs serially.
    if subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True).returncode != 0:
        subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16.argtypes = [P, I64, P]
        lib.oracle_round_bf16.restype = None
        lib.oracle_code.argtypes = [P, I64, I64, I64]
        lib.oracle_code.restype = ctypes.c_int
        lib.oracle_e2m1_value.argtypes = [ctypes.c_int]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_dequant_int4.argtypes = [P, P, P, I64, I64, I64, P]
        lib.oracle_dequant_int4.restype = None
        lib.oracle_dequant_fp4.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_dequant_fp4.restype = None
        lib.oracle_gemm_int4.argtypes = [P, P, P, P, I64, I64, I64, I64, P]
        lib.oracle_gemm_int4.restype = None
        lib.oracle_moe_fp4.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, P,
                                       ctypes.POINTER(ctypes.c_int)]
        lib.oracle_moe_fp4.restype = None
        lib.oracle_gemm_bf16.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_gemm_bf16.restype = None
        lib.oracle_moe_fp4_gemm.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, I64, P,
                                            ctypes.POINTER(ctypes.c_int)]
        lib.oracle_moe_fp4_gemm.restype = None
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_threads.restype = None
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (np.dtype(dtype), a.dtype))
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _zptr(z):
    """Zero points or NULL (symmetric INT4)."""
    return ctypes.c_void_p(None) if z is None else _ptr(z)


def set_threads(n: int) -> None:
    """Threads used by the products (default 1).  Every output element is
    still computed by one thread in the serial order, so results are the
    same for any count; only the timed CPU baseline raises it."""
    _load().oracle_set_threads(int(n))


# ----------------------------------------------------------------- formats

def f16_to_f64(bits: int) -> float:
    """IEEE binary16 bit pattern -> value."""
    return _load().oracle_f16_to_f64(int(bits) & 0xFFFF)


def bf16_to_f64(bits: int) -> float:
    """bfloat16 bit pattern -> value."""
    return _load().oracle_bf16_to_f64(int(bits) & 0xFFFF)


def f64_to_bf16(v: float) -> int:
    """binary64 -> bfloat16 bits, round to nearest even, one rounding."""
    return int(_load().oracle_f64_to_bf16(float(v)))


def round_bf16(y: np.ndarray) -> np.ndarray:
    """Round an array of binary64 values to bfloat16 bit patterns (uint16)."""
    y = _c(np.asarray(y, dtype=np.float64), np.float64)
    out = np.empty(y.shape, dtype=np.uint16)
    _load().oracle_round_bf16(_ptr(y), y.size, _ptr(out))
    return out


def code(qw: np.ndarray, K: int, n: int, k: int) -> int:
    """4-bit code of element (n, k) of a packed [N, K/2] matrix."""
    qw = _c(qw, np.uint8)
    return int(_load().oracle_code(_ptr(qw), K, n, k))


def e2m1_value(c: int) -> float:
    """E2M1 code (0..15) -> value."""
    return float(_load().oracle_e2m1_value(int(c)))


# -------------------------------------------------------------- dequantise

def dequant_int4(qw, s, z, K: int, group: int = 128) -> np.ndarray:
    """W[N, K] (float32) = ((float)q - (float)z) * (float)s per element;
    z=None: symmetric INT4 (z = 8 for every group)."""
    qw = _c(qw, np.uint8)
    s = _c(s, np.uint16)
    z = None if z is None else _c(z, np.uint16)
    N = qw.size // (K // 2)
    _check_int4(qw, s, z, N, K, group)
    W = np.empty((N, K), dtype=np.float32)
    _load().oracle_dequant_int4(_ptr(qw), _ptr(s), _zptr(z), N, K, group, _ptr(W))
    return W


def dequant_fp4(qw, s, K: int, group: int = 32) -> np.ndarray:
    """W[rows, K] (float32) = e2m1(code) * (float)s per element."""
    qw = _c(qw, np.uint8)
    s = _c(s, np.uint16)
    rows = qw.size // (K // 2)
    if K % group or qw.size != rows * (K // 2) or s.size != rows * (K // group):
        raise ValueError("inconsistent FP4 shapes")
    W = np.empty((rows, K), dtype=np.float32)
    _load().oracle_dequant_fp4(_ptr(qw), _ptr(s), rows, K, group, _ptr(W))
    return W


def _check_int4(qw, s, z, N, K, group):
    if K % group or K % 2:
        raise ValueError("K must be a multiple of the group size")
    if qw.size != N * (K // 2):
        raise ValueError("qw has %d bytes, expected %d" % (qw.size, N * (K // 2)))
    G = K // group
    if s.size != N * G or (z is not None and z.size != N * G):
        raise ValueError("s/z must hold N*K/group values")


# ---------------------------------------------------------------- products

def gemm_int4(X, qw, s, z, K: int, group: int = 128) -> np.ndarray:
    """Y[M, N] (float64) = X W^T with INT4 weights; X bfloat16 bits [M, K];
    z=None: symmetric INT4 (z = 8)."""
    X = _c(np.asarray(X).reshape(-1, K), np.uint16)
    qw = _c(qw, np.uint8)
    s = _c(s, np.uint16)
    z = None if z is None else _c(z, np.uint16)
    M = X.shape[0]
    N = qw.size // (K // 2)
    _check_int4(qw, s, z, N, K, group)
    Y = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_int4(_ptr(X), _ptr(qw), _ptr(s), _zptr(z), M, N, K,
                             group, _ptr(Y))
    return Y


def gemv_int4(x, qw, s, z, K: int, group: int = 128) -> np.ndarray:
    """y[N] (float64) for one activation row x (bfloat16 bits [K])."""
    return gemm_int4(np.asarray(x).reshape(1, K), qw, s, z, K, group)[0]


def moe_fp4(x, qw, s, ids, E: int, N: int, K: int, group: int = 32):
    """Y[topk, N] (float64) and the count of ids outside [0, E).

    qw is the [E, N, K/2] expert stack, s the [E, N, K/group] scales and
    ids the expert id of each output row, in order."""
    x = _c(np.asarray(x).reshape(-1), np.uint16)
    qw = _c(qw, np.uint8)
    s = _c(s, np.uint16)
    ids = _c(np.asarray(ids, dtype=np.int32), np.int32)
    if x.size != K or qw.size != E * N * (K // 2) or s.size != E * N * (K // group):
        raise ValueError("inconsistent MoE shapes")
    topk = ids.size
    Y = np.empty((topk, N), dtype=np.float64)
    bad = ctypes.c_int(0)
    _load().oracle_moe_fp4(_ptr(x), _ptr(qw), _ptr(s), _ptr(ids), topk, E, N,
                           K, group, _ptr(Y), ctypes.byref(bad))
    return Y, int(bad.value)


def moe_fp4_gemm(X, qw, s, ids, E: int, N: int, K: int, group: int = 32):
    """Y[M, topk, N] (float64) and the count of ids outside [0, E).

    X: bfloat16 bits [M, K]; ids: [M, topk] expert ids (row (m, j) of Y uses
    expert ids[m, j]); qw the [E, N, K/2] expert stack, s its [E, N, K/group]
    scales."""
    X = _c(np.asarray(X).reshape(-1, K), np.uint16)
    M = X.shape[0]
    ids = _c(np.asarray(ids, dtype=np.int32).reshape(M, -1), np.int32)
    topk = ids.shape[1]
    qw = _c(qw, np.uint8)
    s = _c(s, np.uint16)
    if qw.size != E * N * (K // 2) or s.size != E * N * (K // group):
        raise ValueError("inconsistent MoE shapes")
    Y = np.empty((M, topk, N), dtype=np.float64)
    bad = ctypes.c_int(0)
    _load().oracle_moe_fp4_gemm(_ptr(X), _ptr(qw), _ptr(s), _ptr(ids), M, topk, E, N,
                                K, group, _ptr(Y), ctypes.byref(bad))
    return Y, int(bad.value)


# ------------------------------------------------------ two-pass ablation

def gemm_bf16(X, W, K: int) -> np.ndarray:
    """Y[M, N] (float64) = X W^T for bfloat16 bit arrays X [M, K], W [N, K]
    (the dense second pass of the unfused dequantise-then-GEMM path)."""
    X = _c(np.asarray(X).reshape(-1, K), np.uint16)
    W = _c(np.asarray(W).reshape(-1, K), np.uint16)
    M, N = X.shape[0], W.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_bf16(_ptr(X), _ptr(W), M, N, K, _ptr(Y))
    return Y
