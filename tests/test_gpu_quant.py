"""GPU parity of the quantised matcher (AnnSA-Quant, AnnCA-Quant, TempCache-Quant).

FAST-AR summary (paperlayer.ai) section 5 "ANN Attention" and appendix C
(quantisation precision, 2 to 32 bits); paper.rainbus.top, reproduction
(FAISS, 8-bit by default).  Compared with the oracle (quant_topk_listed,
tempcache_nn_quant_listed), cascaded as in tests/parity.py:
  * the per-query selection (sel_mask) equals the oracle's top-k outside
    listed near-ties at the k-th score, with exactly min(k, n) keys per query;
  * the attention output, computed by the oracle on the GPU's own selection,
    within max 1e-2 / mean 1e-3 (lse within 1e-3);
  * TempCache-Quant decisions bit-exact outside listed ones, and the cache
    state as for the method's merge.
Bits 2, 8 and 16 (two 8-bit-or-less code widths and the 16-bit one); ragged
sizes (197 tokens per frame, 77 prompt tokens, several 64-key tiles and a
partial one).
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import ATT_MAX, ATT_MEAN, Report, cache_to_oracle, check_att, dev, host
from test_gpu_path import _path, build_cache, run_chunk
from workloads import CONFIGS, layer_data

pytestmark = pytest.mark.gpu


def _cfg():
    return CONFIGS[0].replace(dtype="bf16", n_f=197, F=2, past_frames=5, P=77, T=2, B=7, C=900, D=128, H=3,
                              redraw=0.3)


def _mask_bool(mask, n):
    """[..][words] int32 bit rows -> bool [..][n]."""
    m = host(mask).astype(np.int64) & 0xFFFFFFFF
    bits = (m[..., :, None] >> np.arange(32)[None, None, :]) & 1
    return bits.reshape(*m.shape[:-1], -1)[..., :n].astype(bool)


def _check_selection(gpu_sel, allowed, listed, k, what):
    n = allowed.shape[1]
    assert (gpu_sel.sum(axis=1) == min(k, n)).all(), f"{what}: not {min(k, n)} keys per query"
    bad = (gpu_sel != allowed) & ~listed
    assert not bad.any(), f"{what}: {int(bad.sum())} selections differ outside the listed near-ties"
    return int(listed.sum()), int(((gpu_sel != allowed) & listed).sum())


@pytest.mark.parametrize("bits", [2, 8, 16])
def test_annsa_quant_against_oracle(bits):
    from merged_attention_autoregressive_gb300 import fastar_annsa_quant_attention
    cfg = _cfg()
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    build_cache(cfg, d, path, Report(), check=False)
    st = cache_to_oracle(path.cache, cfg.dtype)
    q = d.chunk_q[0]
    qd = dev(q, cfg.dtype)
    words = (cfg.C + 31) // 32
    sel = torch.zeros(cfg.H, cfg.Nq, words, dtype=torch.int32, device="cuda")
    out = torch.zeros(cfg.H, cfg.Nq, cfg.D, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(cfg.H, cfg.Nq, dtype=torch.float32, device="cuda")
    rep = Report()
    for topk in (57, 10 ** 6):
        fastar_annsa_quant_attention(qd, path.cache, cfg.scale, topk, bits, out, lse, sel_mask=sel,
                                     status=path.status)
        torch.cuda.synchronize()
        assert int(path.status.item()) == 0
        o_ref = np.zeros((cfg.H, cfg.Nq, cfg.D))
        lse_ref = np.zeros((cfg.H, cfg.Nq))
        for h in range(cfg.H):
            n = int(st.size[h])
            bias = np.log(np.maximum(st.m[h, :n], 1).astype(np.float64))
            allowed, listed = O.quant_topk_listed(q[h], st.K[h, :n], bias, topk, bits, cfg.scale)
            g = _mask_bool(sel[h], n)
            assert not _mask_bool(sel[h], words * 32)[:, n:].any(), "bits beyond the live slots"
            ln, dn = _check_selection(g, allowed, listed, topk, f"AnnSA-Quant {bits} bits h{h}")
            rep.listed_nn += ln
            rep.differing_listed_nn += dn
            o_ref[h], lse_ref[h] = O.masked_attention(q[h], st.K[h, :n], st.V[h, :n], g, bias, cfg.scale)
        check_att(out, o_ref, f"AnnSA-Quant {bits} bits k {topk}", rep)
        gl = host(lse).astype(np.float64)
        assert np.abs(gl - lse_ref).max() <= 1e-3
    # every key kept: dense attention over the live cache (+ ln m)
    o_all, _ = O.annsa_quant_attention(q, st, 10 ** 6, bits, cfg.scale)
    check_att(out, o_all, f"AnnSA-Quant {bits} bits every key", rep)


@pytest.mark.parametrize("bits", [2, 8])
def test_annca_quant_against_oracle(bits):
    from merged_attention_autoregressive_gb300 import fastar_annca_quant_attention
    cfg = _cfg()
    d = layer_data(cfg)
    q = d.chunk_q[0]
    qd, kp, vp = dev(q, cfg.dtype), dev(d.prompt_k, cfg.dtype), dev(d.prompt_v, cfg.dtype)
    words = (cfg.P + 31) // 32
    sel = torch.zeros(cfg.H, cfg.Nq, words, dtype=torch.int32, device="cuda")
    out = torch.zeros(cfg.H, cfg.Nq, cfg.D, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rep = Report()
    topk = 23
    fastar_annca_quant_attention(qd, kp, vp, cfg.scale, topk, bits, out, sel_mask=sel, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref = np.zeros((cfg.H, cfg.Nq, cfg.D))
    for h in range(cfg.H):
        allowed, listed = O.quant_topk_listed(q[h], d.prompt_k[h], np.zeros(cfg.P), topk, bits, cfg.scale)
        g = _mask_bool(sel[h], cfg.P)
        ln, dn = _check_selection(g, allowed, listed, topk, f"AnnCA-Quant {bits} bits h{h}")
        rep.listed_nn += ln
        rep.differing_listed_nn += dn
        o_ref[h], _ = O.masked_attention(q[h], d.prompt_k[h], d.prompt_v[h], g, np.zeros(cfg.P), cfg.scale)
    check_att(out, o_ref, f"AnnCA-Quant {bits} bits", rep)


@pytest.mark.parametrize("bits", [2, 8, 16])
def test_tempcache_quant_chain(bits):
    """The merge with the quantised search along a short history and one
    chunk (cascaded: decisions outside listed ones, then the cache state),
    with the capacity cut so that eviction runs; the rest of the chunk path
    as for the method."""
    cfg = _cfg().replace(C=500)
    d = layer_data(cfg)
    path = _path(cfg, search=f"quant{bits}")
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)
    assert int(host(path.cache.evicted).sum()) > 0
    print("report", rep)
