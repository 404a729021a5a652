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
