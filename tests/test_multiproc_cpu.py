"""The N > 1 bench path on CPU: two gloo ranks (127.0.0.1) run the replica
set-up, the barrier and the max-over-ranks reduction that bench.py uses."""
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
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    import torch.distributed as dist
    d, r, w, local = bench.dist_setup(None)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(d)
    m = bench.max_over_ranks(d, 1.5 + rank)      # slowest rank's time wins
    out[rank] = m
    bench.barrier(d)
    dist.destroy_process_group()


def test_two_rank_replica_plumbing():
    if torch.cuda.is_available():
        pytest.skip("CPU (gloo) test")
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork after threads exist
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == 2.5
