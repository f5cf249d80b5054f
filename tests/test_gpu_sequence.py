"""A decode step as one call ("Lab 5", sections "CUDA Graph" and "Performance
analysis"): w4a16_linear_sequence launches INT4 linears in order on one
stream, w4a16_graph_create captures the same launches into a CUDA graph.

Each chain below feeds linears from earlier ones' outputs (and overwrites
buffers that earlier linears read).  The oracle runs the same chain on its
own, every intermediate rounded to bfloat16 as the device stores it.

Two kinds of data:
 * exact chains: integer activations, two +-1 weights per row and unit
   scales, so that every product and every intermediate is an exactly
   representable integer; the device must then match the oracle bit for bit
   (the sharp test of launch order and of reads after writes);
 * random chains (the generators' usual data), compared with the tolerance
   of a chain (chain_close below)."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import REL_RMSE_MAX, ELEM_REL_MAX, bf16_to_f64, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu

# (M, N, K, symmetric, source buffer, destination buffer)
CHAIN_M1 = [
    (1, 512, 384, False, "x1", "a"),
    (1, 384, 512, False, "a", "b"),
    (1, 512, 384, True, "b", "a"),      # overwrites a, which the previous op read
    (1, 1000, 512, False, "a", "c"),
]
MIXED = [
    (1, 512, 384, False, "x1", "a"),
    (8, 256, 384, False, "x8", "g"),    # tensor cores, independent of the M = 1 chain
    (1, 384, 512, True, "a", "b"),
    (3, 128, 384, False, "x3", "h"),    # three rows sharing one pass over the weights
    (1, 512, 384, False, "b", "a"),
    (8, 384, 256, True, "g", "g2"),     # consumes the tensor-core output
    (3, 256, 128, False, "h", "h2"),
]
INPUTS = {"x1": (1, 384), "x8": (8, 384), "x3": (3, 384)}


def _weights(chain, seed):
    out = []
    for i, (M, N, K, sym, _, _) in enumerate(chain):
        p = synth.int4_problem(N, K, seed=seed * 100 + i)
        out.append((p["qw"], p["s"], None if sym else p["z"]))
    return out


def _inputs(seed):
    return {k: synth.normal_bf16(synth.Stream(seed * 7 + len(k) + r), (r, K))
            for k, (r, K) in INPUTS.items()}


def _exact_weights(chain, seed):
    """Two entries +-1 per row (the rest 0), scale 1, zero points in 2..13
    (the codes z +- 2 stay in 0..15) or none for the symmetric ops: every
    output is an integer of magnitude at most 2 max|x|."""
    out = []
    for i, (M, N, K, sym, _, _) in enumerate(chain):
        st = synth.Stream(seed * 100 + i)
        G = K // 128
        z = (2 + st.words(N * G) % np.uint64(12)).astype(np.int64).reshape(N, G)
        if sym:
            z[:] = 8
        codes = np.repeat(z, 128, axis=1)
        pick = st.words(4 * N)
        for n in range(N):
            for j in range(2):
                col = int(pick[2 * n + j] % np.uint64(K))
                codes[n, col] += 1 if int(pick[2 * N + 2 * n + j]) & 1 else -1
        qw = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        s = np.ones((N, G), dtype=np.float16).view(np.uint16)
        out.append((qw, s, None if sym else z.astype(np.float16).view(np.uint16)))
    return out


def _exact_inputs(seed):
    """Integer activations in -3..3 (exact in bfloat16)."""
    out = {}
    for k, (r, K) in INPUTS.items():
        v = (synth.Stream(seed * 7 + len(k) + r).words(r * K) % np.uint64(7)).astype(np.float32) - 3.0
        out[k] = (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16).reshape(r, K)
    return out


def _oracle_chain(chain, weights, inputs):
    """Final unrounded output of every destination buffer."""
    bufs = {k: v.copy() for k, v in inputs.items()}
    final = {}
    for (M, N, K, _, src, dst), (qw, s, z) in zip(chain, weights):
        X = bufs[src].reshape(-1)[:M * K].reshape(M, K)
        y = oracle.gemm_int4(X, qw, s, z, K=K)
        bufs[dst] = oracle.round_bf16(y)
        final[dst] = y
    return final


def _device_ops(torch, chain, weights, inputs):
    """Device tensors of the chain: one buffer per name, each op taking an
    exact-sized view of it."""
    cap = {}
    for M, N, K, _, src, dst in chain:
        cap[src] = max(cap.get(src, 0), M * K)
        cap[dst] = max(cap.get(dst, 0), M * N)
    bufs = {k: torch.full((n,), float("nan"), dtype=torch.bfloat16, device="cuda") for k, n in cap.items()}
    for k, v in inputs.items():
        if k in bufs:
            bufs[k][:v.size].copy_(dev_tensor(v.reshape(-1), torch.bfloat16))
    ops = []
    for (M, N, K, _, src, dst), (qw, s, z) in zip(chain, weights):
        ops.append((bufs[src][:M * K], dev_tensor(qw, torch.uint8), dev_tensor(s, torch.float16),
                    None if z is None else dev_tensor(z, torch.float16), bufs[dst][:M * N]))
    return bufs, ops


def chain_close(y_bits, ref, what):
    """Tolerance of a chain of products.  Relative RMSE <= 5e-3, as for one
    product.  Per element |y - ref| <= 2e-2 (|ref| + rms(ref)): the floor is
    the output's RMS, not 1, because both sides round every intermediate to
    bfloat16 and, where the device's binary32 result and the exact value lie
    on opposite sides of a rounding boundary, the next linear receives
    inputs one ulp apart; these differences add up as noise proportional to
    the scale of the outputs (simulated with a 1e-4 device error per linear:
    worst ratio 0.013 over the four-linear chain, against 0.05 with the
    floor 1)."""
    y = bf16_to_f64(y_bits).reshape(ref.shape)
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    rel = float(np.linalg.norm(y - ref)) / max(float(np.linalg.norm(ref)), 1e-300)
    worst = np.abs(y - ref) / (np.abs(ref) + rms)
    i = int(np.argmax(worst))
    assert rel <= REL_RMSE_MAX, "%s: rel RMSE %.3g" % (what, rel)
    assert worst.flat[i] <= ELEM_REL_MAX, "%s: element %d: gpu %r vs oracle %r" % (what, i, y.flat[i], ref.flat[i])


def _shapes(chain):
    return {dst: (M, N) for M, N, K, _, src, dst in chain}


def _check(torch, chain, bufs, final, what):
    shapes = _shapes(chain)
    for name, ref in final.items():
        M, N = shapes[name]
        chain_close(host_bits16(bufs[name][:M * N]).reshape(M, N), ref, "%s buffer %s" % (what, name))


def _check_exact(torch, chain, bufs, final, what):
    shapes = _shapes(chain)
    for name, ref in final.items():
        M, N = shapes[name]
        assert np.array_equal(ref, np.round(ref)) and np.abs(ref).max() <= 256, "inexact construction"
        got = bf16_to_f64(host_bits16(bufs[name][:M * N])).reshape(M, N)
        bad = np.flatnonzero(got != ref)
        assert bad.size == 0, "%s buffer %s: %d elements differ, first %d: gpu %r vs oracle %r" % (
            what, name, bad.size, bad[0], got.flat[bad[0]], ref.flat[bad[0]])


@pytest.mark.parametrize("chain", [CHAIN_M1, MIXED], ids=["m1_chain", "mixed"])
def test_exact_chain_bit_exact_direct_and_graph(chain):
    torch, w4 = cuda_or_skip()
    weights, inputs = _exact_weights(chain, 6), _exact_inputs(6)
    final = _oracle_chain(chain, weights, inputs)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    w4.w4a16_linear_sequence(ops)
    torch.cuda.synchronize()
    _check_exact(torch, chain, bufs, final, "sequence")
    g = w4.w4a16_graph_create(ops)
    try:
        for k, v in bufs.items():
            if k not in INPUTS:
                v.fill_(float("nan"))
        for _ in range(3):
            g.launch()
        torch.cuda.synchronize()
    finally:
        g.destroy()
    assert w4.w4a16_check_device_error() == 0
    _check_exact(torch, chain, bufs, final, "graph")


@pytest.mark.parametrize("chain", [CHAIN_M1, MIXED], ids=["m1_chain", "mixed"])
def test_sequence_matches_oracle_chain(chain):
    torch, w4 = cuda_or_skip()
    weights, inputs = _weights(chain, 1), _inputs(1)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    w4.w4a16_linear_sequence(ops)
    torch.cuda.synchronize()
    assert w4.w4a16_check_device_error() == 0
    _check(torch, chain, bufs, _oracle_chain(chain, weights, inputs), "sequence")


def test_graph_replays_read_current_inputs_and_match_the_sequence():
    torch, w4 = cuda_or_skip()
    chain = MIXED
    weights, inputs = _weights(chain, 2), _inputs(2)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    w4.w4a16_linear_sequence(ops)
    torch.cuda.synchronize()
    direct = {k: host_bits16(v).copy() for k, v in bufs.items()}
    g = w4.w4a16_graph_create(ops)
    try:
        for k, v in bufs.items():          # the replay must rewrite every output
            if k not in INPUTS:
                v.fill_(float("nan"))
        g.launch()
        torch.cuda.synchronize()
        for k, v in bufs.items():          # same kernels, same order: same bits
            assert np.array_equal(host_bits16(v), direct[k]), k
        # the next step's inputs written in place; the graph reads them
        new_inputs = _inputs(3)
        for k, v in new_inputs.items():
            bufs[k][:v.size].copy_(dev_tensor(v.reshape(-1), torch.bfloat16))
        g.launch()
        torch.cuda.synchronize()
        _check(torch, chain, bufs, _oracle_chain(chain, weights, new_inputs), "graph replay")
        once = {k: host_bits16(v).copy() for k, v in bufs.items()}
        for _ in range(50):
            g.launch()
        torch.cuda.synchronize()
        assert w4.w4a16_check_device_error() == 0
        for k, v in bufs.items():
            assert np.array_equal(host_bits16(v), once[k]), k
    finally:
        g.destroy()


def test_one_decoder_layer_at_full_shapes_through_a_graph():
    # the seven linears of one layer of the 48-layer decode step (hidden 3840,
    # 16 query heads and 8 key/value heads of 256, MLP 15360): q, k, v and
    # the MLP's gate and up read the hidden state h; o reads q's output (the
    # attention itself is not on this path); down reads up's output
    torch, w4 = cuda_or_skip()
    H, Q, KV, F = 3840, 4096, 2048, 15360
    chain = [(1, Q, H, False, "h", "q"), (1, KV, H, False, "h", "k"), (1, KV, H, False, "h", "v"),
             (1, H, Q, False, "q", "o"), (1, F, H, False, "h", "gate"), (1, F, H, False, "h", "up"),
             (1, H, F, False, "up", "down")]
    weights = _weights(chain, 4)
    inputs = {"h": synth.normal_bf16(synth.Stream(99), (1, H))}
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    g = w4.w4a16_graph_create(ops)
    try:
        g.launch()
        torch.cuda.synchronize()
    finally:
        g.destroy()
    assert w4.w4a16_check_device_error() == 0
    _check(torch, chain, bufs, _oracle_chain(chain, weights, inputs), "decoder layer")


def test_empty_sequence_launches_nothing():
    torch, w4 = cuda_or_skip()
    w4.w4a16_linear_sequence([])
    torch.cuda.synchronize()


def test_failed_check_launches_nothing():
    torch, w4 = cuda_or_skip()
    chain = CHAIN_M1
    weights, inputs = _weights(chain, 5), _inputs(5)
    bufs, ops = _device_ops(torch, chain, weights, inputs)
    # op 2 gets K = 320, not a multiple of the group: the host check fails
    x, qw, s, z, y = ops[2]
    bad_qw = torch.zeros(qw.shape[0], 160, dtype=torch.uint8, device="cuda")
    bad_s = torch.ones(qw.shape[0] * 2, dtype=torch.float16, device="cuda")
    ops[2] = (bufs["b"][:320], bad_qw, bad_s, None, y)
    with pytest.raises(w4.W4A16Error, match="op 2"):
        w4.w4a16_linear_sequence(ops)
    with pytest.raises(w4.W4A16Error, match="op 2"):
        w4.w4a16_graph_create(ops)
    torch.cuda.synchronize()
    for name in ("a", "b", "c"):
        assert torch.isnan(bufs[name].float()).all(), name
