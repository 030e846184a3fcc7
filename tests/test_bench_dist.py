"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the value is
the tokens of all ranks over the slowest rank's time."""
import os
import socket

import pytest
import torch
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
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    t = bench.max_over_ranks(1.0 + rank, w, torch.device("cpu"))
    n = bench.sum_over_ranks(100.0 * (rank + 1), w, torch.device("cpu"))
    bench.barrier(w)
    out[rank] = (t, n)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_aggregate_max_time_and_total_tokens():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == (2.0, 300.0)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.sum_over_ranks(7.0, 1, torch.device("cpu")) == 7.0
