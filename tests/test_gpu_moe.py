"""Batched-expert FP4 GEMV through the C ABI vs the binary64 oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


def _run(w4, torch, m, ids=None):
    ids = m["ids"] if ids is None else ids
    y = w4.fp4_moe_gemv(dev_tensor(m["x"], torch.bfloat16), dev_tensor(m["qw"], torch.uint8),
                        dev_tensor(m["s"], torch.float16), dev_tensor(ids, torch.int32))
    torch.cuda.synchronize()
    return host_bits16(y)


@pytest.mark.parametrize("E,N,K,topk", [(1, 1, 64, 1), (4, 37, 192, 3), (8, 300, 1024, 8),
                                        (16, 1000, 7168, 6), (3, 64, 16384, 2)])
def test_moe_small_and_ragged(E, N, K, topk):
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_problem(E, N, K, topk, seed=E + N + K)
    ref, bad = oracle.moe_fp4(m["x"], m["qw"], m["s"], m["ids"], E=E, N=N, K=K)
    assert bad == 0
    assert_close(_run(w4, torch, m), ref, "moe")


def test_moe_full_size_config():
    # 64 experts of 4096 x 7168 resident; 6 selected by seeded sampling
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_problem(64, 4096, 7168, 6, seed=0)
    ref, bad = oracle.moe_fp4(m["x"], m["qw"], m["s"], m["ids"], E=64, N=4096, K=7168)
    assert bad == 0
    assert_close(_run(w4, torch, m), ref, "moe full")


def test_moe_first_last_and_repeated_experts():
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_problem(64, 128, 512, 4, seed=4)
    ids = np.array([0, 63, 63, 0], np.int32)
    ref, bad = oracle.moe_fp4(m["x"], m["qw"], m["s"], ids, E=64, N=128, K=512)
    y = _run(w4, torch, m, ids)
    assert_close(y, ref, "moe ids")
    assert np.array_equal(y.reshape(4, 128)[1], y.reshape(4, 128)[2])


def test_moe_out_of_range_id_zero_row_and_status():
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_problem(8, 96, 256, 3, seed=2)
    ids = np.array([2, 8, 5], np.int32)
    assert w4.w4a16_check_device_error() == 0
    y = _run(w4, torch, m, ids).reshape(3, 96)
    assert np.all(y[1] == 0)
    ref, bad = oracle.moe_fp4(m["x"], m["qw"], m["s"], ids, E=8, N=96, K=256)
    assert bad == 1
    assert_close(y, ref, "moe bad id")
    assert w4.w4a16_check_device_error() == 6     # W4A16_ERR_DEVICE, then cleared
    assert w4.w4a16_check_device_error() == 0
