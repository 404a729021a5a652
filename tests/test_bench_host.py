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
