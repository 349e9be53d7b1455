"""The multi-rank timing path of bench.py on CPU ranks (gloo, world size 2):
every rank gets the slowest rank's time, and the whole-job value counts the
work of all ranks (weak scaling: each rank runs its own copy of the workload)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    m = bench.dist_max(times[rank], dist, torch.device("cpu"))
    ws, r, lr = bench.dist_info()
    out[rank] = (m, ws, r, lr)
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_value():
    world = 2
    times = [3.5, 4.25]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), times, out), nprocs=world,
                       start_method="spawn", join=True)
    for rank in range(world):
        m, ws, r, lr = out[rank]
        assert m == max(times) and ws == world and r == rank and lr == rank
    import bench
    assert bench.weak_value(2, 1e12, 4.25) == pytest.approx(2 * 1e12 / 4.25e-3 / 1e12)
