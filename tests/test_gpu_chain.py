"""A chain of M = 1 linears in one persistent launch (w4a16_linear_chain;
"Lab 5", sections "CUDA Graph" and "Performance analysis").

The chain computes what the per-op sequence computes, with the same
arithmetic per row, so its outputs must equal w4a16_linear_sequence's bit for
bit; both are also checked against the oracle run on the same chain.  The
dependency rules (reads after writes, writes after reads and writes) are
exercised by chains whose ops feed each other and overwrite buffers earlier
ops read, by ops with fewer rows than there are CTAs, by chains longer than
one launch holds, and by replays from a CUDA graph.  The scratch must be left
zeroed by every call, also by one whose waits were made to run out."""
import time

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import cuda_or_skip, dev_tensor, host_bits16
from tests.test_gpu_sequence import (CHAIN_M1, _check, _check_exact, _device_ops, _exact_inputs, _exact_weights,
                                     _inputs, _oracle_chain, _weights)

pytestmark = pytest.mark.gpu

def _chain_wide():
    # a: 16 outputs feed op 1 through a 128-long view (the rest of "a2" is input)
    return [
        (1, 16, 384, False, "x1", "a"),
        (1, 384, 128, True, "x1", "b"),
        (1, 3000, 384, False, "x1", "c"),
        (1, 384, 384, False, "b", "x1"),     # overwrites x1, read by ops 0-2
        (1, 7, 384, False, "x1", "d"),       # reads the new x1
        (1, 640, 384, True, "c", "e"),       # reads c, written long before
    ]


def _run_chain(torch, w4, ops, scratch):
    w4.w4a16_linear_chain(ops, scratch)
    torch.cuda.synchronize()


def _scratch_is_zero(torch, scratch):
    return int(torch.count_nonzero(scratch)) == 0


@pytest.mark.parametrize("which", ["m1", "wide"])
def test_chain_equals_sequence_bitwise_and_matches_oracle(which):
    torch, w4 = cuda_or_skip()
    chain = CHAIN_M1 if which == "m1" else _chain_wide()
    weights, inputs = _weights(chain, 11), _inputs(11)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    w4.w4a16_linear_sequence(ops)
    torch.cuda.synchronize()
    direct = {k: host_bits16(v).copy() for k, v in bufs.items()}
    for k, v in bufs.items():                       # fresh inputs, cleared outputs
        if k in inputs:
            v[:inputs[k].size].copy_(dev_tensor(inputs[k].reshape(-1), torch.bfloat16))
        else:
            v.fill_(float("nan"))
    scratch = w4.chain_scratch(len(ops))
    _run_chain(torch, w4, ops, scratch)
    assert w4.w4a16_check_device_error() == 0
    assert _scratch_is_zero(torch, scratch)
    for k, v in bufs.items():
        assert np.array_equal(host_bits16(v), direct[k]), "buffer %s differs from the sequence" % k
    _check(torch, chain, bufs, _oracle_chain(chain, weights, inputs), "chain")


def test_exact_chain_is_bit_exact():
    torch, w4 = cuda_or_skip()
    chain = CHAIN_M1
    weights, inputs = _exact_weights(chain, 6), _exact_inputs(6)
    final = _oracle_chain(chain, weights, inputs)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    scratch = w4.chain_scratch(len(ops))
    for _ in range(3):                              # the scratch is reused as the call left it
        _run_chain(torch, w4, ops, scratch)
    assert _scratch_is_zero(torch, scratch)
    _check_exact(torch, chain, bufs, final, "chain")


def test_chain_longer_than_one_launch():
    """200 ops: two launches (192 + 8), each op reading the previous one's
    output, so the second launch depends on the first through the stream."""
    torch, w4 = cuda_or_skip()
    n = 200
    chain = [(1, 128, 128, i % 3 == 0, "a" if i % 2 == 0 else "b", "b" if i % 2 == 0 else "a") for i in range(n)]
    chain[0] = (1, 128, 128, False, "x0", "b")
    weights = []
    for i, (M, N, K, sym, _, _) in enumerate(chain):   # one +-1 per row: |y| <= max |x|
        st = synth.Stream(800 + i)
        z = np.full((N, K // 128), 8 if sym else 3 + i % 9, dtype=np.int64)
        codes = np.repeat(z, 128, axis=1)
        pick = st.words(2 * N)
        for n_ in range(N):
            codes[n_, int(pick[n_] % np.uint64(K))] += 1 if int(pick[N + n_]) & 1 else -1
        qw = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        s = np.ones((N, K // 128), dtype=np.float16).view(np.uint16)
        weights.append((qw, s, None if sym else z.astype(np.float16).view(np.uint16)))
    st = synth.Stream(8)
    v = (st.words(128) % np.uint64(7)).astype(np.float32) - 3.0
    inputs = {"x0": (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16).reshape(1, 128)}
    final = _oracle_chain(chain, weights, inputs)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    scratch = w4.chain_scratch(n)
    assert scratch.numel() * 4 >= w4.w4a16_linear_chain_scratch_bytes(n)
    _run_chain(torch, w4, ops, scratch)
    assert w4.w4a16_check_device_error() == 0
    assert _scratch_is_zero(torch, scratch)
    last = {chain[-1][5]: final[chain[-1][5]]}
    _check_exact(torch, chain, bufs, last, "long chain")


def test_chain_in_a_cuda_graph_reads_current_inputs():
    torch, w4 = cuda_or_skip()
    chain = _chain_wide()
    weights, inputs = _weights(chain, 12), _inputs(12)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    scratch = w4.chain_scratch(len(ops))
    _run_chain(torch, w4, ops, scratch)             # first call outside the capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            w4.w4a16_linear_chain(ops, scratch, stream=s)
    torch.cuda.synchronize()
    for step in range(3):
        new = _inputs(20 + step)
        bufs["x1"][:new["x1"].size].copy_(dev_tensor(new["x1"].reshape(-1), torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert _scratch_is_zero(torch, scratch)
        _check(torch, chain, bufs, _oracle_chain(chain, weights, new), "graph replay %d" % step)
    assert w4.w4a16_check_device_error() == 0


def test_decoder_layer_at_full_shapes_in_one_launch():
    torch, w4 = cuda_or_skip()
    H, Q, KV, F = 3840, 4096, 2048, 15360
    chain = [(1, Q, H, False, "h", "q"), (1, KV, H, False, "h", "k"), (1, KV, H, False, "h", "v"),
             (1, H, Q, False, "q", "o"), (1, F, H, False, "h", "gate"), (1, F, H, False, "h", "up"),
             (1, H, F, False, "up", "down")]
    weights = _weights(chain, 4)
    inputs = {"h": synth.normal_bf16(synth.Stream(99), (1, H))}
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    scratch = w4.chain_scratch(len(ops))
    _run_chain(torch, w4, ops, scratch)
    assert w4.w4a16_check_device_error() == 0
    _check(torch, chain, bufs, _oracle_chain(chain, weights, inputs), "decoder layer chain")


@pytest.mark.parametrize("flag", ["producers", "consumers"])
def test_chain_timeout_reports_and_leaves_scratch_zero(flag):
    torch, w4 = cuda_or_skip()
    chain = _chain_wide()
    weights, inputs = _weights(chain, 13), _inputs(13)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    scratch = w4.chain_scratch(len(ops))
    w4.w4a16_debug_inject(w4.INJECT_STALL_PIPELINE if flag == "producers" else w4.INJECT_STALL_CONSUMERS)
    try:
        t0 = time.monotonic()
        w4.w4a16_linear_chain(ops, scratch)
        status = w4.w4a16_check_device_error()
        waited = time.monotonic() - t0
    finally:
        w4.w4a16_debug_inject(0)
    assert status == 5, status
    assert 1.5 < waited < 60.0, waited
    assert _scratch_is_zero(torch, scratch)
    for k, v in bufs.items():
        if k in inputs:
            v[:inputs[k].size].copy_(dev_tensor(inputs[k].reshape(-1), torch.bfloat16))
    _run_chain(torch, w4, ops, scratch)
    assert w4.w4a16_check_device_error() == 0
    _check(torch, chain, bufs, _oracle_chain(chain, weights, inputs), "chain after recovery")
