"""bench.py's multi-process plumbing on CPU: two gloo ranks (replicas of the
path, no data-path collective) agree on the barrier and report the maximum
of their step times."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # each replica times its own work; the job's time is the slowest rank's
    got = bench.max_over_ranks(1.5 + rank, w)
    out[rank] = got
    bench.barrier(w)
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU gloo test")
def test_two_gloo_ranks_take_the_max_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}
