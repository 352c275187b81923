"""bench.py's replica path on CPU: two gloo ranks, the job's time is the
slowest rank's and its rate counts every rank's units (the GPU path does the
same over NCCL)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = 2.0 + 3.0 * rank  # rank 1 is the slow one
        mx = bench.max_over_ranks(ms)
        q.put((rank, mx, bench.job_rate(1e9, world, mx)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, rate in res:
        assert mx == 5.0
        assert rate == pytest.approx(2 * 1e9 / 5e-3)


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)
