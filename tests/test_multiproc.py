"""The multi-GPU host logic of bench.py on CPU: world size 2 over gloo.

N GPUs run N independent layers (rank r runs layer r, the data differ per
layer) with no collective on the data path; the only exchange is the
job-time reduction (the slowest rank's time), checked here without a GPU.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from workloads import CONFIGS, layer_data
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.rank_info()
        assert (r, w, local) == (rank, world, rank)
        # the job time is the largest rank time
        out[rank] = bench.job_max(1.5 + rank, w, "cpu")
        # each rank runs its own layer: different data, same shapes
        cfg = CONFIGS[0]
        d = layer_data(cfg, layer=bench.rank_layer(r), chunks=1)
        out[world + rank] = float(np.asarray(d.chunk_k[0], dtype=np.float64).sum())
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 2.5
    assert out[2] != out[3]  # rank 0 and rank 1 ran different layers
