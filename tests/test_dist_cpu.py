"""The benchmark's multi-rank path on CPU: two gloo ranks (127.0.0.1)
combine their step times as the slowest rank's and count every rank's
tokens (weak scaling, no data-path collective)."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, value = bench.combine_ranks(2.0 + rank, 1000, world, torch.device("cpu"))
    dist.barrier()
    out[rank] = (ms, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_slowest_time_and_all_tokens():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == 3.0                      # the slower rank's 3 ms
        assert abs(value - 2000 / 3e-3) < 1e-6  # both ranks' tokens / slowest time


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.combine_ranks(4.0, 500, 1, torch.device("cpu"))
    assert ms == 4.0 and abs(value - 500 / 4e-3) < 1e-9
