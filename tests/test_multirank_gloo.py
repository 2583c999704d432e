"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Every GPU run here has one GPU, so the N>1 path (one replica of the step per rank,
no data-path collective, the job time = the slowest rank) is covered on the host."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 10 + r ms; the job takes the slowest rank's time
        slowest = bench.max_over_ranks(10.0 + rank, world)
        rate = bench.job_rate(1e12, world, slowest, 1e12)
        q.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_job_rate(world):
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(world))
    for rank, slowest, rate in got:
        assert slowest == 10.0 + world - 1
        # 1 TFLOP per rank, world ranks, 11 ms -> world / 0.011 TFLOP/s
        assert abs(rate - world / 0.011) < 1e-6


def test_job_rate_single():
    import bench
    assert bench.job_rate(2e9, 1, 1000.0, 1e9) == 2.0
