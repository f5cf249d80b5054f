"""The chain entry point that allocates nothing (w4a16_linear_chain_noalloc),
called through the C ABI.

Some callers cannot allocate device memory: an engine that gives all of the
GPU to its own memory pool and passes plug-in code only its tensors, or code
that must not risk the device-wide synchronisation cudaMalloc can cause.  For
them the library keeps the chain's completion counters in a built-in device
array instead of caller scratch.  This test checks that entry against the
chain with caller scratch on the same linears, twice in a row (the second
call finds the array as the first left it), and against the oracle.

The file is named to be collected last; it needs nothing from other tests
and passes when run alone in a fresh process."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import ELEM_REL_MAX, REL_RMSE_MAX, bf16_to_f64, cuda_or_skip, dev_tensor, host_bits16

pytestmark = pytest.mark.gpu

# (N, K, symmetric, source buffer, destination buffer): each op after the
# first reads an earlier op's output; "x" is overwritten by op 3 after ops 0-2
# read it
CHAIN = [
    (512, 384, False, "x", "a"),
    (384, 512, True, "a", "b"),
    (640, 384, False, "x", "c"),
    (384, 384, False, "b", "x"),
    (256, 640, False, "c", "d"),
]


def _close(y_bits, ref, what):
    # the chain tolerance of the sequence tests: |y - ref| <= 2e-2 (|ref| +
    # rms(ref)) per element, relative RMSE <= 5e-3
    y = bf16_to_f64(y_bits).reshape(ref.shape)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    rel = float(np.linalg.norm(y - ref)) / max(float(np.linalg.norm(ref)), 1e-300)
    worst = float(np.max(np.abs(y - ref) / (np.abs(ref) + rms)))
    assert rel <= REL_RMSE_MAX and worst <= ELEM_REL_MAX, "%s: rel %.3g worst %.3g" % (what, rel, worst)


def test_noalloc_chain_matches_the_chain_with_scratch_twice():
    torch, w4 = cuda_or_skip()
    weights = []
    for i, (N, K, sym, _, _) in enumerate(CHAIN):
        p = synth.int4_problem(N, K, seed=500 + i)
        weights.append((p["qw"], p["s"], None if sym else p["z"]))
    x0 = synth.normal_bf16(synth.Stream(501), (384,))

    # the oracle on the same chain, every intermediate rounded to bfloat16
    bufs = {"x": x0.copy()}
    final = {}
    for (N, K, _, src, dst), (qw, s, z) in zip(CHAIN, weights):
        y = oracle.gemm_int4(bufs[src].reshape(-1)[:K].reshape(1, K), qw, s, z, K=K)[0]
        bufs[dst] = oracle.round_bf16(y)
        final[dst] = y

    def device_run(noalloc):
        dbufs = {k: torch.full((n,), float("nan"), dtype=torch.bfloat16, device="cuda")
                 for k, n in {"x": 384, "a": 512, "b": 384, "c": 640, "d": 256}.items()}
        dbufs["x"].copy_(dev_tensor(x0, torch.bfloat16))
        ops = [(dbufs[src][:K], dev_tensor(qw, torch.uint8), dev_tensor(s, torch.float16),
                None if z is None else dev_tensor(z, torch.float16), dbufs[dst][:N])
               for (N, K, _, src, dst), (qw, s, z) in zip(CHAIN, weights)]
        arr = w4.w4a16_linear_array(ops)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        if noalloc:
            # straight through the C ABI: ops, count, group, stream
            status = w4.lib().w4a16_linear_chain_noalloc(arr, len(ops), 128, stream)
            assert status == 0, w4.w4a16_last_error_string()
        else:
            scratch = w4.chain_scratch(len(ops))
            w4.w4a16_linear_chain(arr, scratch, count=len(ops))
        torch.cuda.synchronize()
        out = {k: host_bits16(v).copy() for k, v in dbufs.items()}
        del ops, arr
        return out

    with_scratch = device_run(noalloc=False)
    for call in range(2):
        got = device_run(noalloc=True)
        assert w4.w4a16_check_device_error() == 0
        for name, ref in final.items():
            n = ref.size
            _close(got[name][:n], ref, "no-alloc call %d, buffer %s vs oracle" % (call, name))
            _close(got[name][:n], bf16_to_f64(with_scratch[name][:n]),
                   "no-alloc call %d, buffer %s vs the chain with scratch" % (call, name))
