"""Cascaded GPU-vs-oracle comparison of the per-chunk path (used by -m gpu tests).

Each stage is compared, then the oracle continues from the GPU's own output
of that stage, so that a listed near-tie (a hash bit or an NN decision
within 1e-4 of its boundary) cannot cascade into later stages:
  hash codes   bit-exact outside the oracle's margin bits
  bucket CSR   bit-exact against the oracle's CSR of the GPU codes
  TempCache    NN decisions bit-exact outside listed ones; cache K, m,
               codes, last_frame, size and counters bit-exact; V within
               1 ulp of the storage type (bf16) or 1e-6 relative (fp32)
  AnnCA prune  kept lists and counts bit-exact
  attention    max |err| <= 1e-2 and mean |err| <= 1e-3 against the
               oracle on the GPU's own inputs and cache state
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle as O

ATT_MAX, ATT_MEAN = 1e-2, 1e-3
TDT = {"bf16": torch.bfloat16, "f32": torch.float32}
ALL_REPORTS = []  # every Report of the session, summed up at the end of the run (conftest)


@dataclass
class Report:
    """Listed (near-boundary) decisions and value differences of one test:
    they are counted, not failed."""
    listed_hash_bits: int = 0
    differing_listed_bits: int = 0
    listed_nn: int = 0
    differing_listed_nn: int = 0
    v_ulp_diffs: int = 0
    att: dict = field(default_factory=dict)

    def __post_init__(self):
        ALL_REPORTS.append(self)


def dev(x: np.ndarray, dtype: str, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device=device, dtype=TDT[dtype])


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    return t.detach().cpu().numpy()


def check_codes(gpu_codes, x, planes, T, B, rep: Report, what=""):
    g = host(gpu_codes).astype(np.uint32)
    o, margin = O.hash_codes(x, planes, T, B)
    diff = (g ^ o)
    assert not (diff & ~margin).any(), f"{what}: hash bits differ outside the margin " \
        f"({int(((diff & ~margin) != 0).sum())} codes)"
    rep.listed_hash_bits += int(sum(bin(int(v)).count("1") for v in margin[margin != 0]))
    rep.differing_listed_bits += int(sum(bin(int(v)).count("1") for v in diff[diff != 0]))
    return g


def check_csr(gpu_perm, gpu_offsets, codes, nb, sizes=None, what=""):
    p = host(gpu_perm)
    off = host(gpu_offsets)
    H, T, N = codes.shape
    for h in range(H):
        n = N if sizes is None else int(sizes[h])
        for t in range(T):
            op, oo = O.bucket_csr(codes[h, t], nb, n=n)
            np.testing.assert_array_equal(p[h, t, :n], op[:n], err_msg=f"{what} perm h{h} t{t}")
            np.testing.assert_array_equal(off[h, t], oo, err_msg=f"{what} offsets h{h} t{t}")


def cache_to_oracle(cache, dtype: str) -> O.CacheState:
    return O.CacheState(dtype, host(cache.K).astype(np.float64), host(cache.V).astype(np.float64),
                        host(cache.m).astype(np.int64), host(cache.codes).astype(np.uint32),
                        host(cache.last_frame).astype(np.int64), host(cache.size).astype(np.int64),
                        host(cache.inserted).astype(np.int64), host(cache.evicted).astype(np.int64))


def _ulp_bf16(x):
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def check_merge(path, st_before: O.CacheState, k, v, gpu_codes, gpu_match, F, n_f, first_frame,
                tau, dtype, rep: Report, what="", search="prev"):
    """Compare one merge call; returns the oracle state continued from the GPU."""
    st_o, match_o, listed = O.tempcache_merge(st_before, k, v, gpu_codes, F, n_f, first_frame, tau,
                                              search=search)
    gm = host(gpu_match).astype(np.int64)
    bad = (gm != match_o) & ~listed
    assert not bad.any(), f"{what}: {int(bad.sum())} NN decisions differ (first at " \
        f"{np.argwhere(bad)[0].tolist()}: gpu {gm[bad][0]} oracle {match_o[bad][0]})"
    rep.listed_nn += int(listed.sum())
    rep.differing_listed_nn += int(((gm != match_o) & listed).sum())
    if ((gm != match_o) & listed).any():
        st_o, _, _ = O.tempcache_merge(st_before, k, v, gpu_codes, F, n_f, first_frame, tau,
                                       match_override=gm, search=search)
    g = cache_to_oracle(path.cache, dtype)
    for name in ("size", "inserted", "evicted"):
        np.testing.assert_array_equal(getattr(g, name), getattr(st_o, name), err_msg=f"{what} {name}")
    for h in range(g.H):
        n = int(g.size[h])
        np.testing.assert_array_equal(g.K[h, :n], st_o.K[h, :n], err_msg=f"{what} K h{h}")
        np.testing.assert_array_equal(g.m[h, :n], st_o.m[h, :n], err_msg=f"{what} m h{h}")
        np.testing.assert_array_equal(g.codes[h, :, :n], st_o.codes[h, :, :n], err_msg=f"{what} codes h{h}")
        np.testing.assert_array_equal(g.last_frame[h, :n], st_o.last_frame[h, :n],
                                      err_msg=f"{what} last_frame h{h}")
        dv = np.abs(g.V[h, :n] - st_o.V[h, :n])
        if dtype == "bf16":
            assert (dv <= _ulp_bf16(st_o.V[h, :n]) * 1.0001).all(), f"{what} V h{h} beyond 1 ulp"
        else:
            assert (dv <= 1e-6 * np.abs(st_o.V[h, :n]) + 1e-7).all(), f"{what} V h{h}"
        rep.v_ulp_diffs += int((dv > 0).sum())
    assert (g.m[:, :].sum(axis=1) + g.evicted == g.inserted).all(), f"{what} count invariant"
    return g


def check_att(gpu_out, ref, what, rep: Report):
    g = host(gpu_out).astype(np.float64)
    err = np.abs(g - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    rep.att[what] = (mx, mean)
    assert mx <= ATT_MAX and mean <= ATT_MEAN, f"{what}: max {mx:.3g} mean {mean:.3g}"
