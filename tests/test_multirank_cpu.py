"""Host-side logic of the multi-rank benchmark path on CPU with gloo, 2 ranks:
the step time reported is the slowest rank's, and the whole-job rate counts
every rank's rows against it."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        assert bench.dist_env() == (world, rank, rank)
        local_ms = 10.0 + 5.0 * rank  # rank 1 is slower
        ms = bench.reduce_max(local_ms)
        rate = bench.whole_job_rate(1000, world, ms)
        q.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_uses_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate in res:
        assert ms == 15.0
        assert rate == pytest.approx(2 * 1000 / 0.015)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_rate(16384, 1, 53.7) == pytest.approx(16384 / 0.0537)
