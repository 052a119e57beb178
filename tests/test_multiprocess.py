"""The multi-rank host logic of bench.py on CPU (two gloo ranks): the barrier
and the max over ranks that sets the step time of a replicated run (every
rank runs the whole workload on its own GPU; no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(True)
        t = bench.max_over_ranks(1.5 + rank, True)        # per-rank step times (ms)
        out[rank] = t
        bench.barrier(True)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_step_time_is_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn", join=True)
        got = dict(out)
    assert got == {0: 2.5, 1: 2.5}
