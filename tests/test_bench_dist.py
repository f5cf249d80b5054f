"""Host logic of the benchmark's multi-process (replica) mode, on CPU.

Two gloo ranks on 127.0.0.1 check that the timing aggregate is the maximum over
ranks, that the barrier returns on every rank, and that the reference arm runs
on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.dist_barrier()
    got = bench.dist_max(1.5 + rank)
    # rank 1 of the reference arm returns at once without touching the oracle
    rc = bench.run_reference(bench.argparse.Namespace(steps=1, warmup=0, gpus=world)) if rank == 1 else 0
    bench.dist_barrier()
    dist.destroy_process_group()
    out.put((rank, got, rc))


def test_replica_timing_is_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0]
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert [r[1] for r in res] == [2.5, 2.5]
    assert [r[2] for r in res] == [0, 0]


def test_single_process_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.25) == 3.25
    bench.dist_barrier()


@pytest.mark.parametrize("fused", [False, True])
def test_decode_step_structure(fused):
    # the pages' step: 48 layers (40 sliding, 8 global), 328 quantised
    # linears, then the 262144-row vocabulary GEMV (the fused layout stores
    # q|k|v and gate|up as one tensor each: the same weights in 193 launches);
    # every activation buffer is written before it is read, within its
    # storage, and each linear's K is its source's length
    import bench
    ops = bench.decode_step_linears(fused)
    views = bench.decode_step_views(fused)
    assert len(ops) == (193 if fused else 329)
    assert ops[-1] == ("h", "logits", 262144, 3840)
    written = {"h": 3840}
    for src, dst, N, K in ops:
        base, off, n = views[src]
        assert n == K and written.get(base, 0) >= off + K, (src, dst)
        base, off, n = views[dst]
        assert off == 0 and N <= n
        written[base] = max(written.get(base, 0), N)
    # INT4 codes + binary16 scales and zeros of the 328 linears (reading of
    # the pages' 5,705,441,280 bytes, whose breakdown is lost): within 0.5 %
    w = sum(N * K // 2 + 2 * 2 * N * (K // 128) for _, _, N, K in ops[:-1])
    assert w == 5681971200
    assert abs(w - 5705441280) / 5705441280 < 5e-3
    if not fused:
        assert sum(1 for op in ops[:-1] if op[1] == "v") == 40


def test_algorithmic_bytes_of_the_roofline():
    # per launch: packed codes (N K / 2) + binary16 scales and zeros
    # (2 x 2 N K / 128) + the activation (2 K) + the output (2 N)
    import bench
    up, down = bench.gemv_bytes(15360, 3840), bench.gemv_bytes(3840, 15360)
    assert up == 15360 * (1920 + 120) + 7680 + 30720 == 31372800
    assert down == up                     # the same matrix transposed: same total
    assert bench.STEP_BYTES == 2 * 31372800
    assert bench.gemv_bytes(262144, 3840) == 535305728   # the vocabulary GEMV
