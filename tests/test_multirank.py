"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): each
rank times its own batch, the job time is the maximum over ranks and the
throughput counts every rank's tokens (weak scaling, no data-path collective)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    ms = 100.0 + 50.0 * rank                    # rank 1 is the slow one
    got = bench.max_over_ranks(ms)
    tput = bench.job_throughput(131072, 10, world, got)
    out[rank] = (ws, r, local, got, tput)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        ws, r, local, got, tput = out[rank]
        assert (ws, r, local) == (world, rank, rank)
        assert got == 150.0
        assert tput == pytest.approx(2 * 131072 * 10 / 0.150)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_throughput(1000, 4, 1, 2.0) == pytest.approx(2e6)
