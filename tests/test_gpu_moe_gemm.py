"""Batched-expert FP4 GEMM (M tokens x topk experts) through the C ABI vs
the binary64 oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import assert_close, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu


def _run(w4, torch, m, ids=None, scratch=None):
    ids = m["ids"] if ids is None else ids
    Y = w4.fp4_moe_gemm(dev_tensor(m["x"], torch.bfloat16), dev_tensor(m["qw"], torch.uint8),
                        dev_tensor(m["s"], torch.float16), dev_tensor(ids, torch.int32), scratch=scratch)
    torch.cuda.synchronize()
    return host_bits16(Y)


def _ref(m, ids=None):
    ids = m["ids"] if ids is None else ids
    return oracle.moe_fp4_gemm(m["x"], m["qw"], m["s"], ids, E=m["E"], N=m["N"], K=m["K"])


@pytest.mark.parametrize("E,N,K,M,topk", [
    (1, 1, 256, 1, 1),          # one row, one token
    (4, 37, 256, 3, 2),         # ragged N below one 128-row block
    (8, 300, 1024, 16, 8),      # every expert, ragged N over three blocks
    (2, 200, 512, 150, 2),      # 150 rows per expert: tiles of 128 and 22 rows
    (16, 1000, 7168, 40, 6),    # the expert FC's K
    (3, 130, 16384, 5, 3),      # long K (the gather's threads hold 8 blocks of 8 values each)
    (2, 40, 16640, 3, 2),       # longer: the gather reads the row twice
    (5, 200, 768, 9, 3),        # K % 512 == 256: a half last weight stage in every item
    (8, 256, 1280, 20, 4),      # the same after two full stages, several items per CTA
    (1500, 8, 256, 40, 4),      # more experts than the routing CTA's threads: its scans run in two chunks
])
def test_moe_gemm_small_and_ragged(E, N, K, M, topk):
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_batch_problem(E, N, K, M, topk, seed=E + N + K + M)
    ref, bad = _ref(m)
    assert bad == 0
    assert_close(_run(w4, torch, m), ref, "moe gemm")


def test_moe_gemm_one_expert_many_tiles():
    # 300 tokens on one expert of eight: tiles of 128, 128 and 44 rows, and
    # experts with no rows at all
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_batch_problem(8, 160, 512, 300, 1, seed=11)
    ids = np.full((300, 1), 5, np.int32)
    ref, bad = _ref(m, ids)
    assert bad == 0
    assert_close(_run(w4, torch, m, ids), ref, "moe gemm one expert")


def test_moe_gemm_first_last_and_repeated_experts():
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_batch_problem(64, 128, 512, 2, 4, seed=4)
    ids = np.array([[0, 63, 63, 0], [63, 63, 63, 63]], np.int32)
    ref, bad = _ref(m, ids)
    y = _run(w4, torch, m, ids)
    assert_close(y, ref, "moe gemm ids")
    y = y.reshape(2, 4, 128)
    assert np.array_equal(y[0, 1], y[0, 2]) and np.array_equal(y[0, 0], y[0, 3])
    assert all(np.array_equal(y[1, 0], y[1, j]) for j in range(4))


def test_moe_gemm_out_of_range_ids_zero_rows_and_status():
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_batch_problem(8, 96, 256, 3, 2, seed=2)
    ids = np.array([[2, 8], [-1, 5], [7, 0]], np.int32)
    assert w4.w4a16_check_device_error() == 0
    y = _run(w4, torch, m, ids).reshape(3, 2, 96)
    assert np.all(y[0, 1] == 0) and np.all(y[1, 0] == 0)
    ref, bad = _ref(m, ids)
    assert bad == 2
    assert_close(y, ref, "moe gemm bad ids")
    assert w4.w4a16_check_device_error() == 6     # W4A16_ERR_DEVICE, then cleared
    assert w4.w4a16_check_device_error() == 0


def test_moe_gemm_reuses_scratch_without_clearing():
    # two calls in a row on one scratch buffer, different routings; and a
    # buffer one byte short is refused
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_batch_problem(6, 136, 768, 20, 3, seed=8)
    need = w4.fp4_moe_gemm_scratch_bytes(20, 3, 6, 768)
    scratch = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    ids2 = np.ascontiguousarray(m["ids"][::-1])
    for ids in (m["ids"], ids2):
        ref, bad = _ref(m, ids)
        assert_close(_run(w4, torch, m, ids, scratch), ref, "moe gemm scratch reuse")
    with pytest.raises(w4.W4A16Error, match="INVALID_ARG"):
        _run(w4, torch, m, None, scratch[: need - 256])


@pytest.fixture(scope="module")
def full_moe():
    # 64 experts of 4096 x 7168 resident; 128 tokens, 6 experts each
    return synth.fp4_moe_batch_problem(64, 4096, 7168, 128, 6, seed=0)


@pytest.mark.parametrize("M", [16, 128])
def test_moe_gemm_full_size_sampled(full_moe, M):
    # the GPU computes every output; the oracle a sample of tokens and rows
    torch, w4 = cuda_or_skip()
    m = dict(full_moe, x=full_moe["x"][:M], ids=full_moe["ids"][:M], M=M)
    y = _run(w4, torch, m).reshape(M, 6, 4096)
    rng = np.random.default_rng(M)
    toks = np.sort(rng.choice(M, 3, replace=False))
    rows = np.sort(rng.choice(4096, 192, replace=False))
    sub = dict(m, x=m["x"][toks], ids=m["ids"][toks], qw=np.ascontiguousarray(m["qw"][:, rows]),
               s=np.ascontiguousarray(m["s"][:, rows]), N=len(rows), M=3)
    ref, bad = _ref(sub)
    assert bad == 0
    assert_close(y[toks][:, :, rows], ref, "moe gemm full M=%d" % M)


@pytest.mark.parametrize("E,N,K,M,topk", [
    (2, 64, 32768, 3, 2),       # long K: 128 chunks, the weight ring wrapping many times
    (64, 256, 512, 1024, 8),    # 8192 (token, slot) pairs: tiles of 128 rows per expert, several each
    (4096, 64, 256, 4, 2),      # many experts: the routing kernel's per-expert counters (48 KB)
])
def test_moe_gemm_large_sizes(E, N, K, M, topk):
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_batch_problem(E, N, K, M, topk, seed=E + M)
    ref, bad = _ref(m)
    assert bad == 0
    assert_close(_run(w4, torch, m), ref, "moe gemm E=%d M=%d K=%d" % (E, M, K))


def test_moe_gemm_in_a_captured_graph():
    """Caller scratch and device ids: the three launches capture into a graph
    and each replay routes the ids it finds."""
    torch, w4 = cuda_or_skip()
    m = synth.fp4_moe_batch_problem(8, 96, 512, 12, 3, seed=31)
    X = dev_tensor(m["x"], torch.bfloat16)
    qw, s = dev_tensor(m["qw"], torch.uint8), dev_tensor(m["s"], torch.float16)
    ids = dev_tensor(m["ids"], torch.int32)
    Y = torch.empty(12, 3, 96, dtype=torch.bfloat16, device="cuda")
    scratch = torch.empty(w4.fp4_moe_gemm_scratch_bytes(12, 3, 8, 512), dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        w4.fp4_moe_gemm(X, qw, s, ids, Y, scratch)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            w4.fp4_moe_gemm(X, qw, s, ids, Y, scratch)
    for new_ids in (m["ids"], np.ascontiguousarray(m["ids"][:, ::-1])):
        ids.copy_(dev_tensor(new_ids, torch.int32))
        g.replay()
        torch.cuda.synchronize()
        ref, bad = _ref(m, new_ids)
        assert_close(host_bits16(Y), ref, "moe gemm graph replay")
    assert w4.w4a16_check_device_error() == 0
