"""Pins for the CPU oracle, independent of the oracle itself.

Each check compares the oracle with something the pages or mathematics fix:
hand-worked fixtures under tests/golden/, closed forms, brute force on tiny
hand-packed matrices, library routines (numpy float16, torch bfloat16) and the
invariant that the fused product equals dequantise-then-dense-matmul.  The
cases are chosen so that swapping the nibbles, dropping the zero point or the
scale, flipping the sign of (q - z), indexing the group or the row wrongly, or
transposing an operand each fail at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.conftest import read_golden

ONE_BF16 = 0x3F80


def f16(v):
    return int(np.array(v, dtype=np.float16).view(np.uint16))


def bf16_bits(values):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits):
    return np.array([oracle.bf16_to_f64(b) for b in np.asarray(bits).ravel()])


def rand_bf16(rng, shape, scale=1.0):
    return bf16_bits(rng.standard_normal(shape) * scale).reshape(shape)


# ------------------------------------------------------------------ formats

def test_f16_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))
    # sign of zero
    assert math.copysign(1.0, oracle.f16_to_f64(0x8000)) == -1.0


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 65536, size=4096).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]              # finite only
    ref = torch.tensor(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = bf16_vals(bits)
    assert np.array_equal(ref, got)


def test_bf16_rounding_fixture():
    for value, bits in read_golden("bf16_rne_cases.txt"):
        assert oracle.f64_to_bf16(float.fromhex(value)) == int(bits, 16), value


def test_bf16_rounding_matches_torch_on_binary32_values():
    # binary32 inputs are exact in binary64, so one-step rounding must agree
    # with torch's float32 -> bfloat16 conversion (round to nearest even).
    rng = np.random.default_rng(2)
    u = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = bf16_bits(f)
    got = oracle.round_bf16(f.astype(np.float64))
    # torch may produce a different NaN payload; there are none here
    assert np.array_equal(ref, got)


# ---------------------------------------------------------------- unpacking

def test_int4_byte_fixture():
    for row in read_golden("int4_byte_cases.txt"):
        byte, z, s, w_even, w_odd = row
        qw = np.array([[int(byte, 16)]], dtype=np.uint8)
        W = oracle.dequant_int4(qw, np.array([[f16(float(s))]], np.uint16),
                                np.array([[f16(float(z))]], np.uint16), K=2,
                                group=2)
        assert W[0, 0] == float(w_even) and W[0, 1] == float(w_odd), row


def test_nibble_order_hand_packed_row():
    # byte j: low nibble j % 16 (even column), high nibble 15 - j % 16 (odd)
    K = 128
    j = np.arange(K // 2)
    qw = (((15 - j % 16) << 4) | (j % 16)).astype(np.uint8).reshape(1, -1)
    s = np.array([[f16(1.0)]], np.uint16)
    z = np.array([[f16(0.0)]], np.uint16)
    W = oracle.dequant_int4(qw, s, z, K=K, group=128)
    assert np.array_equal(W[0, 0::2], (j % 16).astype(np.float32))
    assert np.array_equal(W[0, 1::2], (15 - j % 16).astype(np.float32))
    assert oracle.code(qw, K, 0, 0) == 0 and oracle.code(qw, K, 0, 1) == 15
    assert oracle.code(qw, K, 0, 6) == 3 and oracle.code(qw, K, 0, 7) == 12


def test_group_boundary_and_row_index():
    # all codes 9; group 0 / group 1 and row 0 / row 1 use distinct s and z
    N, K, g = 2, 256, 128
    qw = np.full((N, K // 2), 0x99, np.uint8)
    z = np.array([[f16(0), f16(15)], [f16(3), f16(8)]], np.uint16)
    s = np.array([[f16(1), f16(0.5)], [f16(2), f16(0.25)]], np.uint16)
    W = oracle.dequant_int4(qw, s, z, K=K, group=g)
    expect = {0: (9.0, -3.0), 1: (12.0, 0.25)}   # (k < 128, k >= 128)
    for n in range(N):
        for k in (0, 126, 127):
            assert W[n, k] == expect[n][0]
        for k in (128, 129, 255):
            assert W[n, k] == expect[n][1]
    # the same values through the product with one-hot activations
    for k in (127, 128):
        x = np.zeros(K, np.uint16)
        x[k] = ONE_BF16
        y = oracle.gemv_int4(x, qw, s, z, K=K, group=g)
        assert np.array_equal(y, W[:, k].astype(np.float64))


def test_e2m1_table_fixture():
    table = {int(c): float(v) for c, v in read_golden("e2m1_table.txt")}
    for c, v in table.items():
        got = oracle.e2m1_value(c)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), c
    # through the packed dequantiser: codes 0..15 in column order, s = 1
    K = 32
    codes = np.arange(K) % 16
    qw = ((codes[1::2] << 4) | codes[0::2]).astype(np.uint8).reshape(1, -1)
    W = oracle.dequant_fp4(qw, np.array([[f16(1.0)]], np.uint16), K=K, group=32)
    assert np.array_equal(W[0], np.array([table[c] for c in codes], np.float32))


def test_fp4_group32_boundary():
    K = 64
    qw = np.full((1, K // 2), 0x22, np.uint8)      # code 2 = 1.0 everywhere
    s = np.array([[f16(3.0), f16(0.5)]], np.uint16)
    W = oracle.dequant_fp4(qw, s, K=K, group=32)
    assert np.all(W[0, :32] == 3.0) and np.all(W[0, 32:] == 0.5)
    assert W[0, 31] == 3.0 and W[0, 32] == 0.5


# ------------------------------------------------------------- closed forms

def _int4(N, K, byte, zval, sval, g=128):
    qw = np.full((N, K // 2), byte, np.uint8)
    z = np.full((N, K // g), f16(zval), np.uint16)
    s = np.full((N, K // g), f16(sval), np.uint16)
    return qw, s, z


def test_all_zero_codes_give_zero():
    rng = np.random.default_rng(3)
    K = 384
    qw, s, z = _int4(5, K, 0x00, 0.0, 1.0)
    s = f16_arr(rng.uniform(0.002, 0.02, size=s.shape))
    y = oracle.gemv_int4(rand_bf16(rng, K), qw, s, z, K=K)
    assert np.all(y == 0.0)


def f16_arr(v):
    return np.asarray(v, dtype=np.float16).view(np.uint16)


def test_all_fifteen_codes_closed_form():
    rng = np.random.default_rng(4)
    K = 384
    c = 3.0 / 256.0                       # exact in FP16
    qw, s, z = _int4(4, K, 0xFF, 0.0, c)
    x = rand_bf16(rng, K)
    y = oracle.gemv_int4(x, qw, s, z, K=K)
    expect = 15.0 * c * math.fsum(bf16_vals(x))
    assert np.allclose(y, expect, rtol=1e-12, atol=1e-12)


def test_code_equal_to_zero_point_gives_zero():
    rng = np.random.default_rng(5)
    K = 256
    qw, s, z = _int4(3, K, 0x77, 7.0, 0.01171875)
    y = oracle.gemv_int4(rand_bf16(rng, K), qw, s, z, K=K)
    assert np.all(y == 0.0)


# Symmetric INT4 ("Lab 5", Quantisation correctness: the symmetric GPTQ
# variant), taken in GPTQ's form with the implicit zero point 8 (z = None).

def test_symmetric_midpoint_codes_give_zero():
    rng = np.random.default_rng(15)
    K = 384
    qw = np.full((4, K // 2), 0x88, np.uint8)     # every code 8
    s = f16_arr(rng.uniform(0.002, 0.02, size=(4, K // 128)))
    y = oracle.gemv_int4(rand_bf16(rng, K), qw, s, None, K=K)
    assert np.all(y == 0.0)
    assert np.all(oracle.dequant_int4(qw, s, None, K=K) == 0.0)


def test_symmetric_extreme_codes_closed_form():
    # codes 15 -> +7 s, codes 0 -> -8 s (two's-complement-like range [-8, 7])
    rng = np.random.default_rng(16)
    K = 256
    c = 5.0 / 512.0                        # exact in FP16
    x = rand_bf16(rng, K)
    sx = math.fsum(bf16_vals(x))
    s = np.full((2, K // 128), f16(c), np.uint16)
    top = oracle.gemv_int4(x, np.full((2, K // 2), 0xFF, np.uint8), s, None, K=K)
    bot = oracle.gemv_int4(x, np.full((2, K // 2), 0x00, np.uint8), s, None, K=K)
    assert np.allclose(top, 7.0 * c * sx, rtol=1e-12, atol=1e-12)
    assert np.allclose(bot, -8.0 * c * sx, rtol=1e-12, atol=1e-12)


def test_symmetric_equals_explicit_zero_point_eight():
    rng = np.random.default_rng(17)
    N, K = 5, 384
    qw = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = f16_arr(rng.uniform(0.002, 0.02, size=(N, K // 128)))
    z8 = np.full((N, K // 128), f16(8.0), np.uint16)
    X = rand_bf16(rng, (2, K))
    assert np.array_equal(oracle.gemm_int4(X, qw, s, None, K=K), oracle.gemm_int4(X, qw, s, z8, K=K))
    assert np.array_equal(oracle.dequant_int4(qw, s, None, K=K), oracle.dequant_int4(qw, s, z8, K=K))


def test_identity_weights_reproduce_activations():
    rng = np.random.default_rng(6)
    K = 128
    codes = np.eye(K, dtype=np.uint8)                  # q[n, n] = 1
    qw = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s = np.full((K, 1), f16(1.0), np.uint16)
    z = np.full((K, 1), f16(0.0), np.uint16)
    X = rand_bf16(rng, (3, K))
    Y = oracle.gemm_int4(X, qw, s, z, K=K)
    assert np.array_equal(Y, bf16_vals(X).reshape(3, K))
    assert np.array_equal(oracle.round_bf16(Y), X)


def test_row_constant_weights_non_square():
    # row n holds code n + 1 everywhere; s[n, g] = g + 1; z = 0
    rng = np.random.default_rng(7)
    N, K = 3, 256
    qw = np.array([[(n + 1) * 17] * (K // 2) for n in range(N)], np.uint8)
    s = np.array([[f16(1.0), f16(2.0)]] * N, np.uint16)
    z = np.zeros((N, 2), np.uint16)
    x = rand_bf16(rng, K)
    xv = bf16_vals(x)
    y = oracle.gemv_int4(x, qw, s, z, K=K)
    base = math.fsum(xv[:128]) + 2.0 * math.fsum(xv[128:])
    assert np.allclose(y, [(n + 1) * base for n in range(N)], rtol=1e-12,
                       atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_fused_equals_dequantise_then_matmul():
    rng = np.random.default_rng(8)
    M, N, K = 3, 37, 384
    qw = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = f16_arr(rng.uniform(0.002, 0.02, size=(N, K // 128)))
    z = f16_arr(rng.integers(0, 16, size=(N, K // 128)).astype(np.float64))
    X = rand_bf16(rng, (M, K))
    Y = oracle.gemm_int4(X, qw, s, z, K=K)
    W = oracle.dequant_int4(qw, s, z, K=K).astype(np.float64)
    ref = bf16_vals(X).reshape(M, K) @ W.T
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    # each output row of the GEMM is the GEMV of that activation row
    for m in range(M):
        assert np.array_equal(Y[m], oracle.gemv_int4(X[m], qw, s, z, K=K))


def test_linearity_in_the_activation():
    rng = np.random.default_rng(9)
    N, K = 11, 256
    qw = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = f16_arr(rng.uniform(0.002, 0.02, size=(N, 2)))
    z = f16_arr(rng.integers(0, 16, size=(N, 2)).astype(np.float64))
    a = rng.integers(-8, 9, size=K).astype(np.float64)
    b = rng.integers(-8, 9, size=K).astype(np.float64)
    ya = oracle.gemv_int4(bf16_bits(a), qw, s, z, K=K)
    yb = oracle.gemv_int4(bf16_bits(b), qw, s, z, K=K)
    yab = oracle.gemv_int4(bf16_bits(a + b), qw, s, z, K=K)
    assert np.allclose(yab, ya + yb, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------- MoE

def _moe_closed_form_case():
    E, N, K, g = 5, 3, 64, 32
    qw = np.full((E, N, K // 2), 0x22, np.uint8)     # E2M1 code 2 = 1.0
    s = np.empty((E, N, K // g), np.uint16)
    for e in range(E):
        for n in range(N):
            for j in range(K // g):
                s[e, n, j] = f16((e + 1) * (n + 1) * (j + 1) / 64.0)
    return E, N, K, g, qw, s


def test_moe_expert_indirection_closed_form():
    rng = np.random.default_rng(10)
    E, N, K, g, qw, s = _moe_closed_form_case()
    x = rand_bf16(rng, K)
    xv = bf16_vals(x)
    base = math.fsum(xv[:32]) + 2.0 * math.fsum(xv[32:])
    ids = np.array([4, 0, 2, 2], np.int32)             # repeats are legal
    Y, bad = oracle.moe_fp4(x, qw, s, ids, E=E, N=N, K=K, group=g)
    assert bad == 0
    for i, e in enumerate(ids):
        for n in range(N):
            assert math.isclose(Y[i, n], (e + 1) * (n + 1) / 64.0 * base,
                                rel_tol=1e-12, abs_tol=1e-12)


def test_moe_out_of_range_ids_zero_rows():
    rng = np.random.default_rng(11)
    E, N, K, g, qw, s = _moe_closed_form_case()
    Y, bad = oracle.moe_fp4(rand_bf16(rng, K), qw, s,
                            np.array([1, 5, -1], np.int32), E=E, N=N, K=K,
                            group=g)
    assert bad == 2
    assert np.all(Y[1:] == 0.0) and np.all(Y[0] != 0.0)


def test_moe_equals_per_expert_dequantise_then_matvec():
    rng = np.random.default_rng(12)
    E, N, K, g = 6, 9, 128, 32
    qw = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    s = f16_arr(rng.uniform(0.01, 0.1, size=(E, N, K // g)))
    x = rand_bf16(rng, K)
    ids = np.array([5, 1, 3], np.int32)
    Y, bad = oracle.moe_fp4(x, qw, s, ids, E=E, N=N, K=K, group=g)
    assert bad == 0
    W = oracle.dequant_fp4(qw, s, K=K, group=g).reshape(E, N, K)
    for i, e in enumerate(ids):
        ref = W[e].astype(np.float64) @ bf16_vals(x)
        assert np.allclose(Y[i], ref, rtol=1e-12, atol=1e-12)


def test_moe_gemm_closed_form_per_token_and_slot():
    """All codes 1.0 and scales (e+1)(n+1)(j+1)/64: every output row (m, slot)
    is (e+1)(n+1)/64 times the token's own weighted sum, e = its expert."""
    rng = np.random.default_rng(13)
    E, N, K, g, qw, s = _moe_closed_form_case()
    M = 3
    X = np.stack([rand_bf16(rng, K) for _ in range(M)])
    ids = np.array([[4, 0], [2, 2], [1, 3]], np.int32)
    Y, bad = oracle.moe_fp4_gemm(X, qw, s, ids, E=E, N=N, K=K, group=g)
    assert bad == 0 and Y.shape == (M, 2, N)
    for m in range(M):
        xv = bf16_vals(X[m])
        base = math.fsum(xv[:32]) + 2.0 * math.fsum(xv[32:])
        for j in range(2):
            for n in range(N):
                assert math.isclose(Y[m, j, n], (ids[m, j] + 1) * (n + 1) / 64.0 * base,
                                    rel_tol=1e-12, abs_tol=1e-12)


def test_moe_gemm_equals_dequantise_then_matmul():
    rng = np.random.default_rng(14)
    E, N, K, g = 5, 7, 128, 32
    qw = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    s = f16_arr(rng.uniform(0.01, 0.1, size=(E, N, K // g)))
    M = 4
    X = np.stack([rand_bf16(rng, K) for _ in range(M)])
    ids = np.array([[0, 4], [3, 1], [1, 1], [2, 0]], np.int32)
    Y, bad = oracle.moe_fp4_gemm(X, qw, s, ids, E=E, N=N, K=K, group=g)
    assert bad == 0
    W = oracle.dequant_fp4(qw, s, K=K, group=g).reshape(E, N, K).astype(np.float64)
    for m in range(M):
        for j in range(2):
            assert np.allclose(Y[m, j], W[ids[m, j]] @ bf16_vals(X[m]), rtol=1e-12, atol=1e-12)


def test_moe_gemm_out_of_range_ids_zero_rows_and_single_token_reduction():
    rng = np.random.default_rng(15)
    E, N, K, g, qw, s = _moe_closed_form_case()
    X = np.stack([rand_bf16(rng, K) for _ in range(2)])
    ids = np.array([[1, 5], [-1, 0]], np.int32)
    Y, bad = oracle.moe_fp4_gemm(X, qw, s, ids, E=E, N=N, K=K, group=g)
    assert bad == 2
    assert np.all(Y[0, 1] == 0.0) and np.all(Y[1, 0] == 0.0)
    assert np.all(Y[0, 0] != 0.0) and np.all(Y[1, 1] != 0.0)
    # one token: the batched definition is the single-token one, bit for bit
    y1, _ = oracle.moe_fp4(X[1], qw, s, np.array([0, 2], np.int32), E=E, N=N, K=K, group=g)
    Yb, _ = oracle.moe_fp4_gemm(X[1:], qw, s, np.array([[0, 2]], np.int32), E=E, N=N, K=K, group=g)
    assert np.array_equal(Yb[0].view(np.uint64), y1.view(np.uint64))


@pytest.mark.parametrize("byte", [0x00, 0x5A, 0xA5, 0xFF])
def test_dequant_fp4_matches_table_for_every_byte_pair(byte):
    table = {int(c): float(v) for c, v in read_golden("e2m1_table.txt")}
    qw = np.full((1, 16), byte, np.uint8)
    W = oracle.dequant_fp4(qw, np.array([[f16(0.5)]], np.uint16), K=32,
                           group=32)
    assert np.all(W[0, 0::2] == table[byte & 15] * 0.5)
    assert np.all(W[0, 1::2] == table[byte >> 4] * 0.5)


# Dense BF16 product (the unfused two-pass path's second pass, "Lab 5",
# section "Triton dequant + cuBLAS").

def test_gemm_bf16_matches_numpy_matmul_non_square():
    rng = np.random.default_rng(21)
    M, N, K = 3, 5, 96
    X = rand_bf16(rng, (M, K))
    W = rand_bf16(rng, (N, K))
    Y = oracle.gemm_bf16(X, W, K=K)
    ref = bf16_vals(X).reshape(M, K).astype(np.float64) @ bf16_vals(W).reshape(N, K).astype(np.float64).T
    assert Y.shape == (M, N)
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_gemm_bf16_identity_weights():
    rng = np.random.default_rng(22)
    K = 64
    W = np.where(np.eye(K, dtype=bool), f16_bf16_one(), 0).astype(np.uint16)
    X = rand_bf16(rng, (4, K))
    assert np.array_equal(oracle.gemm_bf16(X, W, K=K), bf16_vals(X).reshape(4, K))


def f16_bf16_one():
    return 0x3F80  # bfloat16 1.0


def test_two_pass_within_bf16_weight_rounding_of_fused():
    # dequantise -> round W to BF16 -> dense product stays within the BF16
    # rounding bound of the fused result: |d| <= 2^-9 * sum_k |x_k w_k|
    rng = np.random.default_rng(23)
    N, K = 6, 384
    p_qw = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = f16_arr(rng.uniform(0.002, 0.02, size=(N, K // 128)))
    z = f16_arr(rng.integers(0, 16, size=(N, K // 128)).astype(np.float64))
    X = rand_bf16(rng, (2, K))
    Wf = oracle.dequant_int4(p_qw, s, z, K=K)
    Wb = oracle.round_bf16(Wf.astype(np.float64)).reshape(N, K)
    two = oracle.gemm_bf16(X, Wb, K=K)
    fused = oracle.gemm_int4(X, p_qw, s, z, K=K)
    bound = 2.0 ** -9 * (np.abs(bf16_vals(X).reshape(2, K)) @ np.abs(Wf.astype(np.float64)).T)
    assert np.all(np.abs(two - fused) <= bound + 1e-12)
    assert np.any(two != fused)  # the rounding is real


def test_thread_count_does_not_change_results():
    """The oracle's optional threads only spread independent output elements:
    results are bitwise those of the serial loop."""
    p = synth.int4_problem(37, 512, M=3, seed=5)
    m = synth.fp4_moe_problem(6, 40, 256, 4, seed=5)
    ref_g = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=512)
    ref_m, _ = oracle.moe_fp4(m["x"], m["qw"], m["s"], m["ids"], E=6, N=40, K=256)
    try:
        oracle.set_threads(4)
        g4 = oracle.gemm_int4(p["x"], p["qw"], p["s"], p["z"], K=512)
        m4, _ = oracle.moe_fp4(m["x"], m["qw"], m["s"], m["ids"], E=6, N=40, K=256)
    finally:
        oracle.set_threads(1)
    assert np.array_equal(g4.view(np.uint64), ref_g.view(np.uint64))
    assert np.array_equal(m4.view(np.uint64), ref_m.view(np.uint64))
