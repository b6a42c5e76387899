"""bench.py's multi-rank plumbing with two gloo ranks on the CPU: process
group set-up from the torchrun environment variables, the barrier around the
timed region, and the max-over-ranks reduction of each rank's time (the
job's time is the slowest rank's).  One GPU per rank runs an independent
replica of the layer step, so these are the only collectives."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    r, w, local = bench.dist_init(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + rank, w)   # rank 0: 1.5, rank 1: 2.5
    bench.barrier(w)
    out[rank] = t
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        got = dict(out)
    assert codes == [0, 0], codes
    assert got == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench

    assert bench.dist_init(1) == (0, 1, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25
