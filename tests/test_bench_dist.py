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
