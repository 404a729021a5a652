"""Full-size GPU parity of the two largest workloads against the fp64 oracle.

* The long-rollout workload: 200 chunks of the Wan-1.3B-like layer (12
  heads, 3 x 1560 tokens per chunk, 5 % of the keys redrawn per frame) from
  an empty cache of capacity 32,768 per head, on every head.  The cache
  fills up around chunk 134 and evicts from then on.  Every chunk's index
  outputs (query, key and prompt codes, query CSR, NN decisions, the whole
  cache state, cache CSR, kept lists) are compared with the oracle, and the
  attention outputs on 256 sampled rows of every tenth chunk.
* The 14B-like 720p layer: 4 seeded layers of the 40, all 40 heads each,
  every merge call (the 21 past frames in calls of 3, then the chunk) and
  every index output in full; attention on every row of the first layer and
  on 256 sampled rows of the others.
The oracle runs in spawned processes, one group of heads each
(tests/fullsize.py); the comparison is cascaded as in tests/parity.py.
"""
import numpy as np
import pytest
import torch

from fullsize import Team, sum_reports
from parity import Report
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


def _bf(arrs):
    """Stack uint16 bf16 bits [1][n][D] of each head into a device bf16 tensor."""
    a = np.ascontiguousarray(np.concatenate(arrs, axis=0)).view(np.int16)
    return torch.from_numpy(a).cuda().view(torch.bfloat16)


def _publish(team, keys, path, rows=None):
    """Copy the GPU outputs of the last call into each unit's shared arrays."""
    c = path.cache
    host = lambda t: t.detach().cpu().numpy()  # noqa: E731
    live = int(c.size.max())   # rows beyond the live slots are never read
    K = host(c.K[:, :live].view(torch.int16)).view(np.uint16)
    V = host(c.V[:, :live].view(torch.int16)).view(np.uint16)
    vals = {"q_codes": host(path.q_codes), "k_codes": host(path.k_codes), "p_codes": host(path.p_codes),
            "q_perm": host(path.q_perm), "q_off": host(path.q_offsets), "match": host(path.match),
            "m": host(c.m), "codes": host(c.codes), "last_frame": host(c.last_frame),
            "perm": host(c.perm), "offsets": host(c.offsets), "kept_idx": host(path.kept_idx),
            "kept_cnt": host(path.kept_cnt)}
    counts = np.stack([host(c.size).astype(np.int64), host(c.inserted), host(c.evicted)], axis=1)
    if rows is not None:
        r = torch.from_numpy(rows).cuda()
        o_ca = host(path.o_ca.index_select(1, r).float())
        o_sa = host(path.o_sa.index_select(1, r).float())
        lse = host(path.lse.index_select(1, r))
    for i, key in enumerate(keys):
        a = team.shm[key].a
        for name, v in vals.items():
            a[name][...] = v[i]
        a["K"][:live] = K[i]
        a["V"][:live] = V[i]
        a["counts"][...] = counts[i]
        if rows is not None:
            a["rows"][:rows.size] = rows
            a["o_ca"][:rows.size] = o_ca[i]
            a["o_sa"][:rows.size] = o_sa[i]
            a["lse"][:rows.size] = lse[i]


def _path(cfg, H):
    from merged_attention_autoregressive_gb300.path import ChunkPath
    return ChunkPath(H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau, torch.bfloat16)


def _record(rep_sum):
    r = Report()
    r.listed_hash_bits = rep_sum.get("listed_hash_bits", 0)
    r.differing_listed_bits = rep_sum.get("differing_listed_bits", 0)
    r.listed_nn = rep_sum.get("listed_nn", 0)
    r.differing_listed_nn = rep_sum.get("differing_listed_nn", 0)
    r.v_ulp_diffs = rep_sum.get("v_ulp_diffs", 0)
    if rep_sum.get("att_rows"):
        r.att["full-size"] = (rep_sum["att_max"], rep_sum["att_mean_max"])
    return r


def test_rollout_200_chunks_full_capacity_all_heads():
    cfg = CONFIGS[2]
    R = 256
    team = Team()
    keys = [(0, h) for h in range(cfg.H)]
    try:
        for h in range(cfg.H):
            team.open(keys[h], cfg, 0, h, R)
        team.wait_open(keys)
        from workloads import planes
        path = _path(cfg, cfg.H)
        path.planes.copy_(torch.from_numpy(planes(cfg, 0)).to("cuda", torch.bfloat16))
        pr = team.call([(k, ("prompt", k)) for k in keys])
        kp, vp = _bf([p[0] for p in pr]), _bf([p[1] for p in pr])
        reps = []
        evicting = None
        for c in range(cfg.chunks):
            fr = team.call([(k, ("frames", k, cfg.F)) for k in keys])
            k_, v_, q_ = (_bf([f[i] for f in fr]) for i in range(3))
            first = cfg.past_frames + c * cfg.F
            path.step(q_, k_, v_, kp, vp, first)
            torch.cuda.synchronize()
            assert int(path.status.item()) == 0, f"chunk {c}: device status {int(path.status.item())}"
            rows = None
            if c % 10 == 9:
                rows = np.sort(np.random.default_rng(c).choice(cfg.Nq, size=R, replace=False)).astype(np.int64)
            _publish(team, keys, path, rows)
            reps += team.call([(k, ("check", k, first, cfg.F, True, R if rows is not None else 0)) for k in keys])
            if evicting is None and int(path.cache.evicted.sum()) > 0:
                evicting = c
        total = sum_reports(reps)
        print("rollout 200 chunks: eviction from chunk", evicting, "report", total)
        assert int(path.cache.size.min()) == cfg.C, "the cache filled up"
        assert evicting is not None and evicting < cfg.chunks - 20, "and evicted for many chunks"
        assert total["att_rows"] == cfg.H * R * (cfg.chunks // 10)
        _record(total)
    finally:
        team.close()


def test_14b_layers_all_heads():
    base = CONFIGS[4]
    layers = [0, 13, 26, 39]
    R = 256
    team = Team()
    try:
        total_reps = []
        for li, layer in enumerate(layers):
            cfg = base
            all_rows = li == 0
            rows_n = cfg.Nq if all_rows else R
            keys = [(layer, h) for h in range(cfg.H)]
            for h in range(cfg.H):
                team.open(keys[h], cfg, layer, h, rows_n)
            team.wait_open(keys)
            from workloads import planes
            path = _path(cfg, cfg.H)
            path.planes.copy_(torch.from_numpy(planes(cfg, layer)).to("cuda", torch.bfloat16))
            f = 0
            while f < cfg.past_frames:
                nF = min(cfg.F, cfg.past_frames - f)
                fr = team.call([(k, ("frames", k, nF)) for k in keys])
                k_, v_ = _bf([x[0] for x in fr]), _bf([x[1] for x in fr])
                codes, match = path.merge(k_, v_, f, F=nF)
                torch.cuda.synchronize()
                assert int(path.status.item()) == 0
                path.k_codes[:, :, :nF * cfg.n_f].copy_(codes)
                path.match[:, :nF * cfg.n_f].copy_(match)
                _publish(team, keys, path)
                total_reps += team.call([(k, ("check", k, f, nF, False, 0)) for k in keys])
                f += nF
            pr = team.call([(k, ("prompt", k)) for k in keys])
            kp, vp = _bf([p[0] for p in pr]), _bf([p[1] for p in pr])
            fr = team.call([(k, ("frames", k, cfg.F)) for k in keys])
            k_, v_, q_ = (_bf([x[i] for x in fr]) for i in range(3))
            path.step(q_, k_, v_, kp, vp, cfg.past_frames)
            torch.cuda.synchronize()
            assert int(path.status.item()) == 0
            rows = np.arange(cfg.Nq, dtype=np.int64) if all_rows else \
                np.sort(np.random.default_rng(layer).choice(cfg.Nq, size=R, replace=False)).astype(np.int64)
            _publish(team, keys, path, rows)
            total_reps += team.call([(k, ("check", k, cfg.past_frames, cfg.F, True, rows.size)) for k in keys])
            for k in keys:
                team.conns[team.where[k]].send(("close", k))
            team.wait_open(keys)
            for k in keys:
                team.shm.pop(k).close()
            del path
            torch.cuda.empty_cache()
        total = sum_reports(total_reps)
        print("14B-like layers", layers, "x 40 heads: report", total)
        assert total["att_rows"] == base.H * (base.Nq + R * (len(layers) - 1))
        _record(total)
    finally:
        team.close()
