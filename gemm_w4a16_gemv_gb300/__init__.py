"""Python binding of the w4a16 CUDA library (include/w4a16.h).

Argument marshalling only: every entry point checks tensor dtypes, shapes,
devices and contiguity, then calls the C ABI of ``_lib/libw4a16.so`` through
ctypes with raw device pointers and the current CUDA stream.  All arithmetic
happens in the library's CUDA kernels; there is no fallback of any kind.  If
the library has not been built, importing this package succeeds but every
call raises ``RuntimeError`` (build it with ``__graft_entry__.build()``).

Tensors: packed codes are ``torch.uint8``; scales and zero points
``torch.float16``; activations and outputs ``torch.bfloat16``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "w4a16_gemv", "w4a16_gemm", "w4a16_gemm_f16", "fp4_moe_gemv", "fp4_moe_gemm", "fp4_moe_gemm_scratch_bytes",
    "w4a16_dequant", "w4a16_bf16_gemm",
    "w4a16_check_device_error", "w4a16_last_error_string", "w4a16_version",
    "w4a16_debug_inject", "INJECT_STALL_PIPELINE", "INJECT_STALL_CONSUMERS",
    "w4a16_linear", "w4a16_linear_array", "w4a16_linear_sequence", "w4a16_graph_create", "w4a16_graph_launch",
    "w4a16_linear_chain", "w4a16_linear_chain_scratch_bytes", "chain_scratch", "w4a16_linear_chain_noalloc",
    "w4a16_graph_destroy", "W4A16Graph",
    "library_path", "W4A16Error", "STATUS", "FMT_INT4", "FMT_FP4",
    "OUT_F32", "OUT_BF16",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libw4a16.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "MISALIGNED",
          4: "CUDA", 5: "TIMEOUT", 6: "DEVICE"}
FMT_INT4, FMT_FP4 = 0, 1
OUT_F32, OUT_BF16 = 0, 1

# Exported symbols and their ctypes signatures (mirrors include/w4a16.h).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int


class w4a16_linear(ctypes.Structure):
    """One INT4 linear of a sequence (mirrors the C struct)."""
    _fields_ = [("x", ctypes.c_void_p), ("qw", ctypes.c_void_p), ("s", ctypes.c_void_p),
                ("z", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


_OPS = ctypes.POINTER(w4a16_linear)
SIGNATURES = {
    "w4a16_gemv": ([_P, _P, _P, _P, _P, _I64, _I64, _INT, _P], _INT),
    "w4a16_gemm": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P], _INT),
    "w4a16_gemm_f16": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P], _INT),
    "w4a16_bf16_gemm": ([_P, _P, _P, _I64, _I64, _I64, _P], _INT),
    "w4a16_copy": ([_P, _P, _I64, _P], _INT),
    "fp4_moe_gemv": ([_P, _P, _P, _P, _INT, _P, _I64, _I64, _I64, _INT, _P], _INT),
    "fp4_moe_gemm": ([_P, _P, _P, _P, _INT, _INT, _P, _I64, _I64, _I64, _INT, _P, _I64, _P], _INT),
    "fp4_moe_gemm_scratch_bytes": ([_INT, _INT, _I64, _I64], _I64),
    "w4a16_dequant": ([_INT, _P, _P, _P, _P, _INT, _I64, _I64, _INT, _P], _INT),
    "w4a16_linear_sequence": ([_OPS, _INT, _INT, _P], _INT),
    "w4a16_linear_chain": ([_OPS, _INT, _INT, _P, _I64, _P], _INT),
    "w4a16_linear_chain_scratch_bytes": ([_INT], _I64),
    "w4a16_linear_chain_noalloc": ([_OPS, _INT, _INT, _P], _INT),
    "w4a16_graph_create": ([_OPS, _INT, _INT, ctypes.POINTER(ctypes.c_void_p)], _INT),
    "w4a16_graph_launch": ([_P, _P], _INT),
    "w4a16_graph_destroy": ([_P], _INT),
    "w4a16_check_device_error": ([_P], _INT),
    "w4a16_debug_inject": ([ctypes.c_uint], _INT),
    "w4a16_last_error_string": ([], ctypes.c_char_p),
    "w4a16_version": ([], _INT),
}


class W4A16Error(RuntimeError):
    """A nonzero status returned by the library."""

    def __init__(self, status: int, message: str):
        super().__init__("%s (%d): %s" % (STATUS.get(status, "?"), status, message))
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    "libw4a16.so is not built (%s); run __graft_entry__.build()" % _LIB_PATH)
            handle = ctypes.CDLL(_LIB_PATH)
            for name, (argtypes, restype) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = handle
        return _lib


def _check(status: int):
    if status != 0:
        msg = lib().w4a16_last_error_string().decode(errors="replace")
        raise W4A16Error(status, msg)


def _stream(stream, device=None):
    """The stream handle to pass: the given stream, else the current stream
    of `device` (of the current device when None)."""
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t: torch.Tensor, name: str, dtype, numel=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if numel is not None and t.numel() != numel:
        raise ValueError("%s has %d elements, expected %d" % (name, t.numel(), numel))
    return ctypes.c_void_p(t.data_ptr())


def w4a16_gemv(x, qw, s, z, y=None, group: int = 128, stream=None):
    """y[N] = x[K] W^T with INT4 weights qw [N, K/2], s/z [N, K/group];
    z=None: symmetric INT4 (zero point 8)."""
    N = qw.shape[0]
    K = 2 * qw.shape[-1]
    dev = qw.device
    px = _need(x, "x", torch.bfloat16, K, dev)
    pq = _need(qw, "qw", torch.uint8, N * K // 2, dev)
    ps = _need(s, "s", torch.float16, N * (K // group), dev)
    pz = _need(z, "z", torch.float16, N * (K // group), dev) if z is not None else None
    if y is None:
        y = torch.empty(N, dtype=torch.bfloat16, device=dev)
    py = _need(y, "y", torch.bfloat16, N, dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().w4a16_gemv(px, pq, ps, pz, py, N, K, group, _stream(stream, dev)))
    return y


def w4a16_gemm(X, qw, s, z, Y=None, group: int = 128, stream=None):
    """Y[M, N] = X[M, K] W^T with INT4 weights qw [N, K/2], s/z [N, K/group];
    z=None: symmetric INT4 (zero point 8)."""
    return _gemm("w4a16_gemm", X, qw, s, z, Y, group, stream)


def w4a16_gemm_f16(X, qw, s, z, Y=None, group: int = 128, stream=None):
    """w4a16_gemm with binary16 operands (each weight rounded once to
    binary16; see the header for the error bound)."""
    return _gemm("w4a16_gemm_f16", X, qw, s, z, Y, group, stream)


def _gemm(name, X, qw, s, z, Y, group, stream):
    N = qw.shape[0]
    K = 2 * qw.shape[-1]
    M = X.numel() // K
    dev = qw.device
    pX = _need(X, "X", torch.bfloat16, M * K, dev)
    pq = _need(qw, "qw", torch.uint8, N * K // 2, dev)
    ps = _need(s, "s", torch.float16, N * (K // group), dev)
    pz = _need(z, "z", torch.float16, N * (K // group), dev) if z is not None else None
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    pY = _need(Y, "Y", torch.bfloat16, M * N, dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(getattr(lib(), name)(pX, pq, ps, pz, pY, M, N, K, group, _stream(stream, dev)))
    return Y


def w4a16_bf16_gemm(X, W, Y=None, stream=None):
    """Y[M, N] = X[M, K] W[N, K]^T, dense BF16 (the unfused path's GEMM)."""
    N, K = W.shape[0], W.shape[-1]
    M = X.numel() // K
    dev = W.device
    pX = _need(X, "X", torch.bfloat16, M * K, dev)
    pW = _need(W, "W", torch.bfloat16, N * K, dev)
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    pY = _need(Y, "Y", torch.bfloat16, M * N, dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().w4a16_bf16_gemm(pX, pW, pY, M, N, K, _stream(stream, dev)))
    return Y


def fp4_moe_gemv(x, qw, s, expert_ids, y=None, group: int = 32, stream=None):
    """y[topk, N]: row i = x W_{expert_ids[i]}^T, FP4 stack qw [E, N, K/2]."""
    E, N = qw.shape[0], qw.shape[1]
    K = 2 * qw.shape[2]
    topk = expert_ids.numel()
    dev = qw.device
    px = _need(x, "x", torch.bfloat16, K, dev)
    pq = _need(qw, "qw", torch.uint8, E * N * K // 2, dev)
    ps = _need(s, "s", torch.float16, E * N * (K // group), dev)
    pi = _need(expert_ids, "expert_ids", torch.int32, topk, dev)
    if y is None:
        y = torch.empty(topk, N, dtype=torch.bfloat16, device=dev)
    py = _need(y, "y", torch.bfloat16, topk * N, dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().fp4_moe_gemv(px, pq, ps, pi, topk, py, E, N, K, group, _stream(stream, dev)))
    return y


def fp4_moe_gemm_scratch_bytes(M: int, topk: int, E: int, K: int) -> int:
    """Bytes of scratch memory fp4_moe_gemm needs for M tokens x topk."""
    return int(lib().fp4_moe_gemm_scratch_bytes(int(M), int(topk), int(E), int(K)))


def fp4_moe_gemm(X, qw, s, expert_ids, Y=None, scratch=None, group: int = 32, stream=None):
    """Y[M, topk, N]: Y[m, j] = X[m] W_{expert_ids[m, j]}^T for the FP4 stack
    qw [E, N, K/2].  `scratch`: a device tensor of at least
    fp4_moe_gemm_scratch_bytes(M, topk, E, K) bytes (allocated per call when
    None)."""
    E, N = qw.shape[0], qw.shape[1]
    K = 2 * qw.shape[2]
    M = X.numel() // K if K else 0
    topk = expert_ids.numel() // M if M else 0
    dev = qw.device
    pX = _need(X, "X", torch.bfloat16, M * K, dev)
    pq = _need(qw, "qw", torch.uint8, E * N * K // 2, dev)
    ps = _need(s, "s", torch.float16, E * N * (K // group), dev)
    pi = _need(expert_ids, "expert_ids", torch.int32, M * topk, dev)
    if Y is None:
        Y = torch.empty(M, topk, N, dtype=torch.bfloat16, device=dev)
    pY = _need(Y, "Y", torch.bfloat16, M * topk * N, dev)
    need = fp4_moe_gemm_scratch_bytes(M, topk, E, K)
    if scratch is None:
        scratch = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if not isinstance(scratch, torch.Tensor) or scratch.device != dev or not scratch.is_contiguous():
        raise ValueError("scratch must be a contiguous CUDA tensor on %s" % dev)
    nbytes = scratch.numel() * scratch.element_size()
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().fp4_moe_gemm(pX, pq, ps, pi, M, topk, pY, E, N, K, group,
                                  ctypes.c_void_p(scratch.data_ptr()), nbytes, _stream(stream, dev)))
    return Y


def w4a16_dequant(fmt: int, qw, s, z=None, out=None, out_dtype: int = OUT_F32,
                  group=None, stream=None):
    """Dequantised weights [rows, K] (float32 or bfloat16) -- debug entry."""
    K = 2 * qw.shape[-1]
    rows = qw.numel() // (K // 2)
    if group is None:
        group = 128 if fmt == FMT_INT4 else 32
    dev = qw.device
    pq = _need(qw, "qw", torch.uint8, rows * K // 2, dev)
    ps = _need(s, "s", torch.float16, rows * (K // group), dev)
    pz = _need(z, "z", torch.float16, rows * (K // group), dev) if z is not None else None
    odt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
    if out is None:
        out = torch.empty(rows, K, dtype=odt, device=dev)
    po = _need(out, "out", odt, rows * K, dev)
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().w4a16_dequant(fmt, pq, ps, pz, po, out_dtype, rows, K, group, _stream(stream, dev)))
    return out


def w4a16_linear_array(ops, group: int = 128):
    """ctypes array of w4a16_linear from (X, qw, s, z, Y) tuples (z may be
    None), each checked as w4a16_gemm checks its tensors.  The array holds
    raw addresses only: the caller keeps the tensors alive while it is used."""
    arr = (w4a16_linear * max(1, len(ops)))()
    for i, (X, qw, s, z, Y) in enumerate(ops):
        N = qw.shape[0]
        K = 2 * qw.shape[-1]
        M = X.numel() // K
        dev = qw.device
        who = "op %d " % i
        arr[i].x = _need(X, who + "x", torch.bfloat16, M * K, dev)
        arr[i].qw = _need(qw, who + "qw", torch.uint8, N * K // 2, dev)
        arr[i].s = _need(s, who + "s", torch.float16, N * (K // group), dev)
        arr[i].z = _need(z, who + "z", torch.float16, N * (K // group), dev) if z is not None else None
        arr[i].y = _need(Y, who + "y", torch.bfloat16, M * N, dev)
        arr[i].M, arr[i].N, arr[i].K = M, N, K
    return arr


def w4a16_linear_sequence(ops, group: int = 128, stream=None, count=None):
    """Launch the INT4 linears `ops` = [(X, qw, s, z, Y), ...] in order on
    one stream (each op's X is read after the previous op has finished).
    `ops` may also be an array from w4a16_linear_array, with `count` ops."""
    if isinstance(ops, ctypes.Array):
        if ops._type_ is not w4a16_linear:
            raise TypeError("ops must be an array of w4a16_linear")
        arr, n = ops, len(ops) if count is None else int(count)
        if not 0 <= n <= len(ops):
            raise ValueError("count %d outside 0..%d (the array's length)" % (n, len(ops)))
        dev = torch.cuda.current_device()  # raw addresses: the caller's current device
    else:
        arr, n = w4a16_linear_array(ops, group), len(ops)
        dev = ops[0][1].device if ops else torch.cuda.current_device()
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().w4a16_linear_sequence(arr, n, group, _stream(stream, dev)))


def w4a16_linear_chain_scratch_bytes(count: int) -> int:
    """Bytes of scratch memory w4a16_linear_chain needs for `count` ops."""
    return int(lib().w4a16_linear_chain_scratch_bytes(int(count)))


def chain_scratch(count: int, device=None) -> torch.Tensor:
    """A zeroed scratch buffer (int32) for chains of up to `count` ops."""
    n = (w4a16_linear_chain_scratch_bytes(count) + 3) // 4
    return torch.zeros(max(n, 1), dtype=torch.int32, device=device if device is not None else "cuda")


def w4a16_linear_chain(ops, scratch, group: int = 128, stream=None, count=None):
    """The M = 1 INT4 linears `ops` = [(x, qw, s, z, y), ...] (or an array
    from w4a16_linear_array with `count` ops) in one persistent launch,
    computing what w4a16_linear_sequence computes.  `scratch`: a zeroed
    device tensor of at least w4a16_linear_chain_scratch_bytes(count)
    bytes (see chain_scratch), left zeroed by every call."""
    if isinstance(ops, ctypes.Array):
        if ops._type_ is not w4a16_linear:
            raise TypeError("ops must be an array of w4a16_linear")
        arr, n = ops, len(ops) if count is None else int(count)
        if not 0 <= n <= len(ops):
            raise ValueError("count %d outside 0..%d (the array's length)" % (n, len(ops)))
        dev = scratch.device
    else:
        arr, n = w4a16_linear_array(ops, group), len(ops)
        dev = ops[0][1].device if ops else scratch.device
    if not isinstance(scratch, torch.Tensor) or not scratch.is_cuda or scratch.device != dev:
        raise ValueError("scratch must be a CUDA tensor on %s" % dev)
    if not scratch.is_contiguous():
        raise ValueError("scratch must be contiguous")
    nbytes = scratch.numel() * scratch.element_size()
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().w4a16_linear_chain(arr, n, group, ctypes.c_void_p(scratch.data_ptr()), nbytes,
                                        _stream(stream, dev)))


def w4a16_linear_chain_noalloc(ops, group: int = 128, stream=None, count=None):
    """w4a16_linear_chain with the library's built-in counters instead of
    caller scratch: nothing is allocated (for callers that may not allocate
    device memory).  At most 4032 linears; calls that can overlap on the GPU
    race on the shared counters, so keep them on one stream."""
    if isinstance(ops, ctypes.Array):
        if ops._type_ is not w4a16_linear:
            raise TypeError("ops must be an array of w4a16_linear")
        arr, n = ops, len(ops) if count is None else int(count)
        if not 0 <= n <= len(ops):
            raise ValueError("count %d outside 0..%d (the array's length)" % (n, len(ops)))
        dev = torch.cuda.current_device()
    else:
        arr, n = w4a16_linear_array(ops, group), len(ops)
        dev = ops[0][1].device if ops else torch.cuda.current_device()
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().w4a16_linear_chain_noalloc(arr, n, group, _stream(stream, dev)))


class W4A16Graph:
    """Handle of a captured linear sequence (w4a16_graph_create).  Keeps the
    tensors of its ops alive: the graph holds their addresses."""

    def __init__(self, handle, tensors, device):
        self._h = handle
        self._tensors = tensors
        self.device = device

    def launch(self, stream=None):
        w4a16_graph_launch(self, stream)

    def destroy(self):
        if self._h is not None:
            h, self._h = self._h, None
            _check(lib().w4a16_graph_destroy(h))
            self._tensors = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def w4a16_graph_create(ops, group: int = 128) -> W4A16Graph:
    """Capture the linear sequence `ops` once into a CUDA graph on the
    current device; replay it with w4a16_graph_launch."""
    arr = w4a16_linear_array(ops, group)
    h = ctypes.c_void_p()
    dev = ops[0][1].device if ops else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):  # the graph is captured on the current device
        _check(lib().w4a16_graph_create(arr, len(ops), group, ctypes.byref(h)))
    return W4A16Graph(h, [t for op in ops for t in op if t is not None], dev)


def w4a16_graph_launch(graph: W4A16Graph, stream=None) -> None:
    """Enqueue one replay of a captured sequence on the stream."""
    if graph._h is None:
        raise ValueError("graph has been destroyed")
    with torch.cuda.device(graph.device):
        _check(lib().w4a16_graph_launch(graph._h, _stream(stream, graph.device)))


def w4a16_graph_destroy(graph: W4A16Graph) -> None:
    graph.destroy()


def w4a16_copy(dst: torch.Tensor, src: torch.Tensor, stream=None, device=None) -> torch.Tensor:
    """dst <- src (the same number of bytes, both contiguous) by one kernel on
    `device` (the CUDA tensor's device; `device` when both are host
    tensors): a CUDA tensor or a pinned host tensor on either side."""
    for name, t in (("dst", dst), ("src", src)):
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a torch.Tensor" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
        if not t.is_cuda and t.numel() > 0 and not t.is_pinned():
            raise ValueError("%s: a host tensor must be pinned" % name)
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst has %d bytes, src %d" % (nbytes, src.numel() * src.element_size()))
    devs = {t.device for t in (dst, src) if t.is_cuda}
    if len(devs) > 1:
        raise ValueError("dst and src are on different devices")
    dev = devs.pop() if devs else torch.device(device if device is not None else "cuda")
    with torch.cuda.device(dev):  # the library launches on the current device
        _check(lib().w4a16_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nbytes,
                                _stream(stream, dev)))
    return dst


def w4a16_check_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status."""
    return int(lib().w4a16_check_device_error(_stream(stream)))


INJECT_STALL_PIPELINE = 1
INJECT_STALL_CONSUMERS = 2


def w4a16_debug_inject(flags: int = 0) -> None:
    """Test-only: make every later GEMV/MoE/GEMM launch on the current device
    issue no stage of its pipeline (flags=1), or take no stage that its
    producers issue (flags=2), so that its bounded waits run out (after about
    2 s) and the device status reports a timeout; flags=0 restores normal
    operation."""
    _check(lib().w4a16_debug_inject(int(flags)))


def w4a16_last_error_string() -> str:
    return lib().w4a16_last_error_string().decode(errors="replace")


def w4a16_version() -> int:
    return int(lib().w4a16_version())
