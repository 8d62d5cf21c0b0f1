"""The multi-GPU bookkeeping of bench.py on CPU ranks (gloo, world size 2).

With N GPUs every rank steps its own unit (independent problems, weak scaling);
the only collective is the max of the timings over ranks, and the job's value
is the sum of all ranks' bytes over that time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank])
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == [2.0, 10.0]


def test_job_value_is_weak_scaling_sum():
    import bench

    one = bench.job_gbs(1_151_068_224, 1, 0.2)
    four = bench.job_gbs(1_151_068_224, 4, 0.2)
    assert four == pytest.approx(4 * one)
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]     # no process group: identity
