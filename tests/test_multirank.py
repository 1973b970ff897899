"""The multi-rank path of bench.py on the CPU: two gloo ranks (world size 2), each timing its own
replica; the line reports the slowest rank's time and the pairs of both ranks. No GPU involved."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slow = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        torch.distributed.barrier()
        q.put((rank, slow, bench.whole_job_gpairs(world, 10 ** 9, 4, slow)))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, value in out:
        assert slow == 2.5  # the max over ranks, seen identically by every rank
        assert value == pytest.approx(2 * 1e9 * 4 / 2.5 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
    assert bench.whole_job_gpairs(1, 2 * 10 ** 9, 1, 2.0) == 1.0
