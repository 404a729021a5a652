"""The multi-GPU host logic of bench.py on CPU: world size 2 over gloo.

Under torchrun each rank runs its share of the chunk: by default the heads
[r H / N, (r+1) H / N) of every layer (each GPU owns its heads' cache slices;
heads share nothing on the path, so there is no collective on the data
path), or whole layers r, r + N, ...  The only exchange is the job-time
reduction (the slowest rank's time).  Checked here without a GPU: the
partition covers every (layer, head) of the chunk exactly once for both
modes and several world sizes, each rank's share of the inputs is exactly
those heads of the full layer (the data do not depend on the split), and the
job time is the largest rank time.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cfg():
    from workloads import CONFIGS
    return CONFIGS[4].replace(H=4, n_f=24, D=64, past_frames=2, P=8, C=128, layers=3, clusters=4)


def _digest(t):
    return [float(x) for x in t.double().sum(dim=(1, 2))]


@pytest.mark.parametrize("mode", ["heads", "layers"])
@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_shard_covers_every_unit_once(mode, world):
    import bench
    cfg = _cfg()
    if (mode == "heads" and world > cfg.H) or (mode == "layers" and world > cfg.layers):
        with pytest.raises(ValueError):
            bench.shard(cfg, 0, world, mode)
        return
    seen = []
    for r in range(world):
        layers, heads = bench.shard(cfg, r, world, mode)
        assert heads == list(range(heads[0], heads[-1] + 1))  # contiguous head slices
        seen += [(lay, h) for lay in layers for h in heads]
    assert sorted(seen) == [(lay, h) for lay in range(cfg.layers) for h in range(cfg.H)]


def _worker(rank, world, port, mode, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.rank_info()
        assert (r, w, local) == (rank, world, rank)
        # the job time is the largest rank time
        out[(mode, "job", rank)] = bench.job_max(1.5 + rank, w, "cpu")
        cfg = _cfg()
        layers, heads = bench.shard(cfg, r, w, mode)
        # the rank's inputs: its heads of each of its layers
        mine = {}
        for lay in layers:
            src = bench.LayerSource(cfg, lay, heads, device="cpu")
            k, v, q = src.frames(cfg.F)
            kp, vp = src.prompt()
            assert k.shape == (len(heads), cfg.F * cfg.n_f, cfg.D) and kp.shape == (len(heads), cfg.P, cfg.D)
            for i, h in enumerate(heads):
                mine[(lay, h)] = (_digest(k[i:i + 1]), _digest(q[i:i + 1]), _digest(kp[i:i + 1]))
        gathered = [None] * w
        dist.all_gather_object(gathered, mine)
        if rank == 0:
            allu = {}
            for g in gathered:
                assert not (set(g) & set(allu)), "a unit ran on two ranks"
                allu.update(g)
            out[(mode, "units")] = allu
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["heads", "layers"])
def test_two_ranks_gloo(mode):
    import bench
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, mode, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    assert out[(mode, "job", 0)] == out[(mode, "job", 1)] == 2.5
    units = out[(mode, "units")]
    cfg = _cfg()
    assert sorted(units) == [(lay, h) for lay in range(cfg.layers) for h in range(cfg.H)]
    # every unit's inputs equal that head of the whole layer drawn on one rank
    for lay in range(cfg.layers):
        src = bench.LayerSource(cfg, lay, list(range(cfg.H)), device="cpu")
        k, v, q = src.frames(cfg.F)
        kp, vp = src.prompt()
        for h in range(cfg.H):
            want = (_digest(k[h:h + 1]), _digest(q[h:h + 1]), _digest(kp[h:h + 1]))
            assert units[(lay, h)] == want, (lay, h)
    # different layers and heads draw different data
    assert units[(0, 0)] != units[(1, 0)] and units[(0, 0)] != units[(0, 1)]
