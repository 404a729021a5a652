"""GPU parity of the mean-key representative (TempCache ablation).

FAST-AR summary (paperlayer.ai), appendix C, compares last-key, mean-key and
medoid-key representatives of a group of corresponding keys.  The library's
mean-key mode (fastar_tempcache_merge_rep with FASTAR_REP_MEAN) keeps the
count-weighted mean key of each group and re-hashes it.  Each merge call
(one frame) is compared with the oracle run from the GPU's own cache state
before the call (so that a one-ulp difference of a stored mean cannot
cascade): NN decisions bit-exact outside listed near-ties; sizes, counts,
last_frame and counters bit-exact; K and V within one ulp of the storage
type; every live group's codes equal to the hash of its stored key outside
margin bits.  A three-frame call must equal three one-frame calls exactly.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import Report, _ulp_bf16, cache_to_oracle, check_att, check_csr, dev, host
from workloads import CONFIGS, layer_data

pytestmark = pytest.mark.gpu


def _path(cfg, rep="mean"):
    from merged_attention_autoregressive_gb300.path import ChunkPath
    p = ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau,
                  dtype={"bf16": torch.bfloat16, "f32": torch.float32}[cfg.dtype], rep=rep)
    return p


def _close(a, b, dtype):
    if dtype == "bf16":
        return np.abs(a - b) <= _ulp_bf16(b) * 1.0001
    return np.abs(a - b) <= 1e-6 * np.abs(b) + 1e-7


def _merge_and_check(path, st, k, v, f, cfg, planes, rep: Report):
    codes, match = path.merge(dev(k, cfg.dtype), dev(v, cfg.dtype), f, F=1)
    torch.cuda.synchronize()
    assert int(path.status.item()) == 0
    gc = host(codes).astype(np.uint32)
    oc, margin = O.hash_codes(k, planes, cfg.T, cfg.B)
    assert not ((gc ^ oc) & ~margin).any()
    gm = host(match).astype(np.int64)
    st_o, match_o, listed = O.tempcache_merge(st, k, v, gc, 1, cfg.n_f, f, cfg.tau, rep="mean",
                                              planes=planes, B=cfg.B)
    bad = (gm != match_o) & ~listed
    assert not bad.any(), f"frame {f}: {int(bad.sum())} NN decisions differ"
    rep.listed_nn += int(listed.sum())
    if ((gm != match_o) & listed).any():
        st_o, _, _ = O.tempcache_merge(st, k, v, gc, 1, cfg.n_f, f, cfg.tau, match_override=gm,
                                       rep="mean", planes=planes, B=cfg.B)
    g = cache_to_oracle(path.cache, cfg.dtype)
    for name in ("size", "inserted", "evicted"):
        np.testing.assert_array_equal(getattr(g, name), getattr(st_o, name), err_msg=f"frame {f} {name}")
    for h in range(g.H):
        n = int(g.size[h])
        np.testing.assert_array_equal(g.m[h, :n], st_o.m[h, :n])
        np.testing.assert_array_equal(g.last_frame[h, :n], st_o.last_frame[h, :n])
        assert _close(g.K[h, :n], st_o.K[h, :n], cfg.dtype).all(), f"frame {f} K h{h}"
        assert _close(g.V[h, :n], st_o.V[h, :n], cfg.dtype).all(), f"frame {f} V h{h}"
        rep.v_ulp_diffs += int((g.K[h, :n] != st_o.K[h, :n]).sum())
        hc, hm = O.hash_codes(g.K[h:h + 1, :n], planes, cfg.T, cfg.B)
        assert not ((hc[0] ^ g.codes[h, :, :n]) & ~hm[0]).any(), f"frame {f} codes h{h}"
    assert (g.m.sum(axis=1) + g.evicted == g.inserted).all()
    check_csr(path.cache.perm, path.cache.offsets, g.codes, 1 << cfg.B, g.size, f"frame {f} CSR")
    return g


def _rollout(cfg, frames):
    d = layer_data(cfg, chunks=1)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    rep = Report()
    merged = 0
    for f in range(frames):
        st = _merge_and_check(path, st, d.past_k[f], d.past_v[f], f, cfg, d.planes, rep)
        merged = max(merged, int((st.m > 1).sum()))
    assert merged > 0, "some groups should merge"
    return d, path, st


def test_meankey_bf16_tensor_path():
    """12 frames of 300 keys, D 128 bf16 (tensor-core NN with the candidates
    staged from the cache every frame), 2 tables x 8 bits, C 2048; then one
    chunk's attention over the mean-key cache against the oracle."""
    cfg = CONFIGS[1].replace(H=2, n_f=300, F=1, past_frames=12, C=2048, redraw=0.3, P=64)
    d, path, st = _rollout(cfg, cfg.past_frames)
    q = d.chunk_q[0]
    path.step(dev(q, cfg.dtype), dev(d.chunk_k[0], cfg.dtype), dev(d.chunk_v[0], cfg.dtype),
              dev(d.prompt_k, cfg.dtype), dev(d.prompt_v, cfg.dtype), cfg.past_frames)
    torch.cuda.synchronize()
    assert int(path.status.item()) == 0
    g = cache_to_oracle(path.cache, cfg.dtype)
    qc = host(path.q_codes).astype(np.uint32)
    o_sa, _ = O.annsa_attention(q, qc, g, cfg.scale)
    check_att(path.o_sa, o_sa, "AnnSA over the mean-key cache", Report())


def test_meankey_fp32_simt_path():
    """The tiny fp32 D 64 layer (CUDA-core NN reading the cache's keys)."""
    cfg = CONFIGS[0].replace(redraw=0.3)
    _rollout(cfg, cfg.past_frames)


def test_meankey_three_frame_call_equals_one_frame_calls():
    cfg = CONFIGS[1].replace(H=2, n_f=300, F=3, past_frames=9, C=2048, redraw=0.3)
    d = layer_data(cfg, chunks=0)
    a, b = _path(cfg), _path(cfg)
    for p in (a, b):
        p.planes.copy_(dev(d.planes, cfg.dtype))
    for f0 in range(0, cfg.past_frames, 3):
        k = np.concatenate(d.past_k[f0:f0 + 3], axis=1)
        v = np.concatenate(d.past_v[f0:f0 + 3], axis=1)
        a.merge(dev(k, cfg.dtype), dev(v, cfg.dtype), f0, F=3)
        for f in range(f0, f0 + 3):
            b.merge(dev(d.past_k[f], cfg.dtype), dev(d.past_v[f], cfg.dtype), f, F=1)
    torch.cuda.synchronize()
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    for name in ("K", "V", "m", "codes", "last_frame", "size", "inserted", "evicted", "offsets"):
        assert torch.equal(getattr(a.cache, name), getattr(b.cache, name)), name
    assert int((a.cache.m > 1).sum()) > 0
