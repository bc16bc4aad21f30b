"""Host logic of bench.py's multi-replica run on CPU: two gloo ranks, the
timed total reduced to the slowest rank, and a distinct batch per replica
(weak scaling, no collective on the data path)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                 # rank 1 is the slower one
        got = bench.max_over_ranks(mine, torch.device("cpu"), dist)
        out[rank] = (got, bench.replica_seed(7, rank))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world,
                       join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] != out[1][1]


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5, torch.device("cpu"), None) == 3.5
