"""bench.py's multi-rank host logic on CPU with the gloo backend (world size 2):
rendezvous from the torchrun environment variables, the barrier, the
max-over-ranks time and the whole-job aggregate.  Replicas share nothing on
the data path, so no collective other than these timing reductions exists."""
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


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    seconds = 1.0 + rank          # rank 1 is the slow one
    slowest = bench.max_over_ranks(seconds, w)
    value = bench.aggregate_value(100.0, w, slowest)
    q.put((rank, slowest, value))
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(100.0 * 2 / 2.0)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_value(10.0, 1, 2.0) == 5.0
