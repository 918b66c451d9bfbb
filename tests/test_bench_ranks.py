"""The multi-rank plumbing of bench.py on CPU: two gloo ranks, no GPU.

bench.py runs one independent replica per GPU (the path does not shard) and
combines ranks only for the report: the job time is the maximum over ranks and
the work is the sum.  These checks run that reduction over two processes.
"""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.5, 40.0][rank]                 # per-rank times of the timed region
    tokens = [85.0, 85.0][rank]             # each replica's work
    out[rank] = (bench.max_over_ranks(world, ms), bench.sum_over_ranks(world, tokens))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_the_summed_work():
    port = 29500 + (os.getpid() % 1000)
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1] == (40.0, 170.0)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1, 3.5) == 3.5 and bench.sum_over_ranks(1, 7.0) == 7.0
