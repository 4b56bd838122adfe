"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): the
timing reduction takes the slowest rank and the whole-job rate sums every
rank's tokens.  The data path itself has no collective (independent
replicas), so nothing else crosses ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank]
        got = bench.max_over_ranks(mine)
        rate = bench.aggregate_rate(32 * 100, world, got[0])
        q.put((rank, got, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_rate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [2.0, 10.0]
        assert rate == pytest.approx(32 * 100 * 2 / 2.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]
    assert bench.aggregate_rate(3200, 1, 2.0) == 1600.0
