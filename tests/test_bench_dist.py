"""bench.py's multi-rank host logic (replicas: barrier + max-over-ranks timing)
on two gloo ranks on the CPU; no data-path collective exists to test."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist(world)
    assert d.pg is not None and d.world == world and d.rank == rank
    d.barrier()
    q.put((rank, d.max(float(10 * (rank + 1)))))
    d.close()


def test_two_rank_max_timing_over_gloo():
    if torch.cuda.is_available():
        pytest.skip("this test exercises the CPU (gloo) path")
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(0, 20.0), (1, 20.0)]
