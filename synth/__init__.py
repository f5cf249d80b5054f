"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws numbers: it holds none of the dequantise or product
arithmetic.  Every tensor comes from one counter-free stream of 64-bit words
(numpy's PCG64 bit generator, raw output, which is fixed by its published
definition and does not depend on numpy's distribution code), mapped by the
explicit formulas below, in the fixed order qw, s, z, x, expert ids.

Mappings (the workloads' distributions):
  * 4-bit codes: uniform over 0..15 -- each raw word supplies 8 bytes, i.e. 16
    independent uniform nibbles, stored little-endian;
  * uniform FP16 in [lo, hi]: u = (w >> 11) * 2^-53, v = lo + (hi - lo) * u,
    rounded to binary16;
  * integer-valued FP16 in [0, 15]: w >> 60;
  * N(0, 1) BF16: Box-Muller on two uniforms in (0, 1], cosine branch and sine
    branch used in turn, rounded to binary32 and then to bfloat16 (nearest,
    ties to even on the bits);
  * expert ids: partial Fisher-Yates over 0..E-1 with index i + (w % (E - i)).

Tensors are returned as numpy arrays of raw bit patterns (uint8 packed codes,
uint16 for FP16/BF16, int32 ids) so both sides see identical bytes.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "Stream", "packed_codes", "uniform_f16", "int_f16", "normal_bf16",
    "sample_experts", "int4_problem", "fp4_moe_problem", "fp4_moe_batch_problem", "CONFIGS",
]


class Stream:
    """A seeded stream of raw 64-bit words."""

    def __init__(self, seed: int = 0):
        self._bg = np.random.PCG64(seed)

    def words(self, n: int) -> np.ndarray:
        if n <= 0:
            return np.zeros(0, dtype=np.uint64)
        return self._bg.random_raw(n).astype("<u8", copy=False)


def packed_codes(st: Stream, rows: int, K: int) -> np.ndarray:
    """uint8 [rows, K/2]: two uniform 4-bit codes per byte."""
    nbytes = rows * (K // 2)
    w = st.words((nbytes + 7) // 8)
    return w.view(np.uint8)[:nbytes].reshape(rows, K // 2)


def uniform_f16(st: Stream, shape, lo: float, hi: float) -> np.ndarray:
    """FP16 bit patterns of lo + (hi - lo) * U[0, 1)."""
    n = int(np.prod(shape))
    u = (st.words(n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    v = lo + (hi - lo) * u
    return v.astype(np.float16).view(np.uint16).reshape(shape)


def int_f16(st: Stream, shape) -> np.ndarray:
    """FP16 bit patterns of integers uniform over 0..15."""
    n = int(np.prod(shape))
    v = (st.words(n) >> np.uint64(60)).astype(np.float64)
    return v.astype(np.float16).view(np.uint16).reshape(shape)


def normal_bf16(st: Stream, shape) -> np.ndarray:
    """BF16 bit patterns of N(0, 1) samples (Box-Muller)."""
    n = int(np.prod(shape))
    pairs = (n + 1) // 2
    w = st.words(2 * pairs)
    u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    v = np.empty(2 * pairs, dtype=np.float64)
    v[0::2] = r * np.cos(t)
    v[1::2] = r * np.sin(t)
    f = v[:n].astype(np.float32).view(np.uint32)
    rounded = (f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16).reshape(shape)


def sample_experts(st: Stream, E: int, topk: int) -> np.ndarray:
    """topk distinct ids from 0..E-1, uniformly, in sampling order."""
    perm = np.arange(E, dtype=np.int64)
    w = st.words(topk)
    for i in range(topk):
        j = i + int(w[i] % np.uint64(E - i))
        perm[i], perm[j] = perm[j], perm[i]
    return perm[:topk].astype(np.int32)


def int4_problem(N: int, K: int, group: int = 128, M: int = 1, seed: int = 0,
                 s_range=(0.002, 0.02)) -> dict:
    """INT4 asymmetric group-quantised weights and BF16 activations.

    qw uint8 [N, K/2]; s, z FP16 bits [N, K/group]; x BF16 bits [M, K]."""
    st = Stream(seed)
    G = K // group
    qw = packed_codes(st, N, K)
    s = uniform_f16(st, (N, G), *s_range)
    z = int_f16(st, (N, G))
    x = normal_bf16(st, (M, K))
    return {"qw": qw, "s": s, "z": z, "x": x, "N": N, "K": K, "M": M,
            "group": group}


def fp4_moe_problem(E: int, N: int, K: int, topk: int, group: int = 32,
                    seed: int = 0, s_range=(0.01, 0.1)) -> dict:
    """FP4 E2M1 expert stack, per-group FP16 scales, one BF16 token.

    qw uint8 [E, N, K/2]; s FP16 bits [E, N, K/group]; x BF16 bits [K];
    ids int32 [topk]."""
    st = Stream(seed)
    qw = packed_codes(st, E * N, K).reshape(E, N, K // 2)
    s = uniform_f16(st, (E, N, K // group), *s_range)
    x = normal_bf16(st, (K,))
    ids = sample_experts(st, E, topk)
    return {"qw": qw, "s": s, "x": x, "ids": ids, "E": E, "N": N, "K": K,
            "topk": topk, "group": group}


def fp4_moe_batch_problem(E: int, N: int, K: int, M: int, topk: int, group: int = 32,
                          seed: int = 0, s_range=(0.01, 0.1)) -> dict:
    """FP4 E2M1 expert stack, per-group FP16 scales and M BF16 tokens, each
    routed to topk distinct experts.

    qw uint8 [E, N, K/2]; s FP16 bits [E, N, K/group]; X BF16 bits [M, K];
    ids int32 [M, topk] (row m: the experts of token m, sampled without
    replacement)."""
    st = Stream(seed)
    qw = packed_codes(st, E * N, K).reshape(E, N, K // 2)
    s = uniform_f16(st, (E, N, K // group), *s_range)
    X = normal_bf16(st, (M, K))
    ids = np.stack([sample_experts(st, E, topk) for _ in range(M)]).astype(np.int32)
    return {"qw": qw, "s": s, "x": X, "ids": ids, "E": E, "N": N, "K": K, "M": M,
            "topk": topk, "group": group}


# The five workloads: Gemma4-12B-shaped INT4 decode/prefill linears and a
# DeepSeek-V4-shaped FP4 expert FC (shapes only; weights are synthetic).
CONFIGS = {
    "gemv_3840x3840": {"kind": "gemv", "N": 3840, "K": 3840},
    "gemv_up_15360x3840": {"kind": "gemv", "N": 15360, "K": 3840},
    "gemv_down_3840x15360": {"kind": "gemv", "N": 3840, "K": 15360},
    "gemv_vocab_262144x3840": {"kind": "gemv", "N": 262144, "K": 3840},
    "gemm_m128_15360x3840": {"kind": "gemm", "M": 128, "N": 15360, "K": 3840},
    "gemm_m2048_15360x3840": {"kind": "gemm", "M": 2048, "N": 15360, "K": 3840},
    "moe_fp4_64x4096x7168_top6": {"kind": "moe", "E": 64, "N": 4096,
                                  "K": 7168, "topk": 6},
}
