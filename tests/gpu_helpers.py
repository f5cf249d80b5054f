"""Helpers shared by the GPU parity tests: device copies and the tolerance."""
import numpy as np
import pytest

# Tolerance for every floating-point product (GEMV, GEMM, MoE): relative RMSE
# over the output tensor and a per-element bound, against the binary64 oracle.
REL_RMSE_MAX = 5e-3
ELEM_REL_MAX = 2e-2


def cuda_or_skip():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_w4a16_gemv_gb300 as w4
    w4.lib()  # fail loudly (RuntimeError) if the library is not built
    return torch, w4


def dev_tensor(a, dtype, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).view(dtype).to(device)


def host_bits16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(y_bits, ref, what=""):
    """GPU bfloat16 output vs the unrounded binary64 oracle."""
    y = bf16_to_f64(y_bits).reshape(ref.shape)
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    denom = max(float(np.linalg.norm(ref)), 1e-300)
    rel = float(np.linalg.norm(y - ref)) / denom
    worst = np.abs(y - ref) / (np.abs(ref) + 1.0)
    i = int(np.argmax(worst))
    assert rel <= REL_RMSE_MAX, "%s: rel RMSE %.3g" % (what, rel)
    assert worst.flat[i] <= ELEM_REL_MAX, "%s: element %d: gpu %r vs oracle %r" % (
        what, i, y.flat[i], ref.flat[i])
    return rel
