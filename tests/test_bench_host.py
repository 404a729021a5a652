"""Host-side pieces of bench.py, checked on CPU.

The allowed-pair count that the bench's effective TFLOP/s rests on (an
inclusion-exclusion over the LSH tables from joint code histograms) equals
the brute-force count of the oracle's allowed mask, and the oracle's timing
team (spawned processes, one (layer, head) unit each) runs and reports a
per-chunk figure consistent with its own step times.
"""
import numpy as np
import pytest
import torch

import oracle as O


@pytest.mark.parametrize("T,B", [(1, 3), (2, 3), (3, 2), (4, 2)])
def test_pairs_union_equals_bruteforce(T, B):
    import bench
    rng = np.random.default_rng(T * 10 + B)
    H, Nq, C = 3, 57, 41
    qc = rng.integers(0, 1 << B, size=(H, T, Nq)).astype(np.int32)
    cc = rng.integers(0, 1 << B, size=(H, T, C)).astype(np.int32)
    sizes = np.array([41, 17, 0], dtype=np.int32)
    total, by_table = bench._pairs_union(torch.from_numpy(qc), torch.from_numpy(cc), torch.from_numpy(sizes), B)
    want, want_t = 0, [0] * T
    for h in range(H):
        n = int(sizes[h])
        allowed = O.annsa_allowed(qc[h].astype(np.uint32), cc[h][:, :n].astype(np.uint32))
        want += int(allowed.sum())
        seen = np.zeros_like(allowed)
        for t in range(T):
            hit = (qc[h, t][:, None] == cc[h, t, :n][None, :]) & ~seen
            want_t[t] += int(hit.sum())
            seen |= hit
    assert total == want and by_table == want_t


def test_oracle_team_times_units():
    import bench
    from workloads import CONFIGS
    cfg = CONFIGS[0].replace(n_f=64, past_frames=2, P=16, layers=2, H=2)
    ob = bench.oracle_baseline(cfg, 2, 1)
    assert ob["cores"] >= 1 and ob["kind"] == "oracle"
    units = cfg.layers * cfg.H
    assert ob["value"] == pytest.approx(ob["ms_per_step"] * units / ob["cores"])
    assert ob["unit_ms_mean"] > 0 and ob["ms_per_step"] >= ob["unit_ms_mean"] * 0.5


def test_rollout_flatness_rule():
    """The rollout's flatness verdict: a flat series with one outlier chunk
    stays flat (the spread is judged on the 95th percentile); a series whose
    latency grows by 2 % per 100 chunks is not, nor is one with a few slow
    chunks in the last 50, nor one whose device memory changes; the trend is
    in percent of the mean per 100 chunks, and with the live-group counts
    given it is judged over the chunks at capacity, after the fill."""
    import bench
    rng = np.random.default_rng(7)
    base = list(0.6 + 0.005 * rng.standard_normal(200))
    mem = [1000] * 200
    spike = base.copy()
    spike[190] = 0.6 * 1.3
    r = bench.flatness(spike, mem)
    assert r["flat"] and r["max_over_median_last50"] > 1.25 and r["p95_over_median_last50"] < 1.05
    trend = [x * (1 + 0.0002 * i) for i, x in enumerate(base)]  # +0.02 % per chunk
    r = bench.flatness(trend, mem)
    assert not r["flat"] and 1.5 < r["slope_last100_pct_of_mean_per_100_chunks"] < 2.5
    slow = base.copy()
    for i in (160, 170, 180, 190):  # 4 of the last 50 chunks 30 % slower: above the 95th percentile
        slow[i] *= 1.3
    assert not bench.flatness(slow, mem)["flat"]
    assert bench.flatness(base, mem)["flat"]
    assert not bench.flatness(base, mem[:-1] + [1001])["flat"]
    # a cache that fills until chunk 140 (latency rising with it), flat after
    fill = [0.3 + 0.3 * min(i, 140) / 140 + 0.003 * rng.standard_normal() for i in range(200)]
    live = [min(1000 * (i + 1), 140_000) for i in range(200)]
    r = bench.flatness(fill, mem, live, 140_000)
    assert r["slope_last100_pct_of_mean_per_100_chunks"] > 5.0
    assert r["trend_window"] == "chunks at capacity" and r["chunks_at_capacity"] == 61
    assert abs(r["slope_at_capacity_pct_of_mean_per_100_chunks"]) < 1.0 and r["flat"]
    # fewer than 50 chunks at capacity: the last 100 chunks decide
    r = bench.flatness(fill, mem, live, 170_000)
    assert r["trend_window"] == "last 100 chunks" and not r["flat"]


def test_layer_work_counts_follow_the_oracle():
    """The work model behind every roofline fraction, on the CPU: for a
    small chain merged by the oracle frame by frame, the NN flops are
    2 D n_f per candidate, the candidates of a frame being the groups the
    previous frame refreshed (counted here from the oracle's cache state);
    the AnnSA flops are 4 D per pair the oracle's mask allows; the kept
    count is the oracle's prune; and the merge bytes count every slot the
    chunk's frames wrote."""
    import types
    import bench
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[0].replace(H=2, n_f=40, F=3, past_frames=3, P=24, T=2, B=4, C=200, redraw=0.3)
    d = layer_data(cfg)
    H, D, T, n_f, F, C, nb = cfg.H, cfg.D, cfg.T, cfg.n_f, cfg.F, cfg.C, 1 << cfg.B
    st = O.CacheState.empty(H, C, D, T, cfg.dtype)
    for f in range(cfg.past_frames):
        st, _, _ = O.tempcache_merge(st, d.past_k[f], d.past_v[f], O.hash_codes(d.past_k[f], d.planes, T, cfg.B)[0],
                                     1, n_f, f, cfg.tau)
    snap = {"last_frame": torch.from_numpy(st.last_frame.copy()), "size": torch.from_numpy(st.size.copy())}
    first = cfg.past_frames
    k, v, q = d.chunk_k[0], d.chunk_v[0], d.chunk_q[0]
    kc = O.hash_codes(k, d.planes, T, cfg.B)[0]
    matches, want_nn, touched = [], 0, 0
    for fi in range(F):
        sl = slice(fi * n_f, (fi + 1) * n_f)
        live = np.arange(C)[None] < st.size[:, None]
        want_nn += 2 * D * n_f * int(((st.last_frame == first + fi - 1) & live).sum())
        st, mt, _ = O.tempcache_merge(st, k[:, sl], v[:, sl], kc[:, :, sl], 1, n_f, first + fi, cfg.tau)
        matches.append(np.asarray(mt))
        touched += int((st.last_frame == first + fi).sum())
    qc = O.hash_codes(q, d.planes, T, cfg.B)[0]
    pc = O.hash_codes(d.prompt_k, d.planes, T, cfg.B)[0]
    kept_idx, kept_cnt = O.annca_prune(qc, pc, F, n_f)
    q_perm, _ = O.bucket_csr(qc, nb)
    offs = np.stack([O.bucket_csr(st.codes[h], nb, int(st.size[h]))[1] for h in range(H)])
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a).astype(np.int32))  # noqa: E731
    cache = types.SimpleNamespace(size=t32(st.size), codes=t32(st.codes), offsets=t32(offs))
    path = types.SimpleNamespace(H=H, C=C, B=cfg.B, cache=cache, kept_cnt=t32(kept_cnt),
                                 match=t32(np.concatenate(matches, axis=1)), q_codes=t32(qc), q_perm=t32(q_perm))
    w = bench.layer_work(cfg, path, snap)
    assert w["flops"]["merge"] == want_nn and w["kern"]["nn_tc"]["flops"] == want_nn
    pairs = sum(int(O.annsa_allowed(qc[h], st.codes[h][:, :int(st.size[h])]).sum()) for h in range(H))
    assert w["flops"]["annsa"] == 4 * D * pairs and w["stats"]["allowed_pairs"] == pairs
    assert w["stats"]["kept"] == int(np.asarray(kept_cnt).sum())
    assert w["stats"]["n_live"] == int(st.size.sum())
    # apply: the frames' k and v read, each refreshed group's old value read,
    # and K, V, m, last_frame and codes written for every slot written
    e = 2 if cfg.dtype == "bf16" else 4
    groups = sum(len(np.unique(mt[h][mt[h] >= 0])) for mt in matches for h in range(H))
    assert w["kern"]["apply"]["bytes"] == (F * 2 * H * n_f * D * e + groups * D * e
                                           + touched * (2 * D * e + 8 + T * 4))
