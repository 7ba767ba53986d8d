"""The multi-rank bench logic on CPU: two gloo ranks, barrier + max over ranks of
the step time, and the whole-job value (ranks x tokens / slowest rank's time)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench._dist()
    assert (ws, r, local) == (world, rank, rank)
    bench._barrier(ws)
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    worst = bench._max_over_ranks(ms, ws, torch.device("cpu"))
    out[rank] = worst
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1] == 15.0
    # whole-job throughput from the slowest rank: 2 ranks x 8192 tokens / 15 ms
    assert abs(world * 8192 / (15.0 / 1e3) - 1092266.67) < 1
