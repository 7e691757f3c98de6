"""The benchmark's multi-rank plumbing on CPU with the gloo backend at world
size 2: the max-over-ranks reduction of the timings, and the reference arm
printing one line from rank 0 only (the other ranks exit without work)."""
import io
import os
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        reduced = bench.max_over_ranks(10.0 + 5.0 * rank)
        buf = io.StringIO()
        args = type("A", (), dict(workload="dit_1p3b", steps=1, warmup=0, gpus=world))()
        # rank 0 would time the oracle; any other rank must return at once and print nothing
        rc = 0
        if rank != 0:
            with redirect_stdout(buf):
                rc = bench.run_reference(args)
        q.put((rank, reduced, rc, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rank0_only_reference():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in procs:
        rank, reduced, rc, printed = q.get(timeout=120)
        out[rank] = (reduced, rc, printed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 15.0
    assert out[1][1] == 0 and out[1][2] == ""


def test_max_over_ranks_without_a_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
