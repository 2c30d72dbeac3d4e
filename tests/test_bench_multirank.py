"""bench.py's multi-rank helpers on CPU with the gloo backend (world size 2).

Under torchrun every rank runs the same workload on its own GPU (independent
problems, no collective on the data path); the only cross-rank steps are the
barrier, the max of the per-rank step time and the sum of the units
processed. These run here as two gloo processes on 127.0.0.1.
"""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    ws, r, local = bench._dist()
    assert (ws, r, local) == (world, rank, rank)
    pg = bench._init_dist(ws, use_cuda=False)
    try:
        cpu = torch.device("cpu")
        # per-rank step times and units; the job's value is the units of all
        # ranks over the slowest rank's time
        ms = bench.reduce_max(pg, [2.0, 3.5][rank], cpu)
        units = bench.reduce_sum(pg, [1000.0, 1000.0][rank], cpu)
        pg.barrier()
        out[rank] = (ms, units)
    finally:
        dist.destroy_process_group()


def test_reductions_over_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world,
             join=True)
    assert out[0] == out[1] == (3.5, 2000.0)


def test_single_process_needs_no_group():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench._init_dist(1, use_cuda=False) is None
    cpu = torch.device("cpu")
    assert bench.reduce_max(None, 1.25, cpu) == 1.25
    assert bench.reduce_sum(None, 7.0, cpu) == 7.0
