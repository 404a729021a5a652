"""GPU parity of the denoising steps of a chunk (ChunkPath.denoise_step).

FAST-AR analysis (paper.rainbus.top), limitations: sparse attention is off
for the first 30 % of a chunk's denoising steps; FAST-AR summary
(paperlayer.ai), related work: each chunk is denoised conditioned on the
history.  Every step is compared with the oracle on the GPU's own codes and
on the cache as it was before the step: a step before the last attends the
cache together with its own keys and must leave the cache untouched; the
last step merges its keys and attends the merged cache.  Attention within
max 1e-2 / mean 1e-3, kept lists and counts bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import Report, cache_to_oracle, check_att, check_codes, check_merge, dev, host
from workloads import CONFIGS, denoise_steps, layer_data

pytestmark = pytest.mark.gpu


def _setup(cfg):
    from merged_attention_autoregressive_gb300.path import ChunkPath
    d = layer_data(cfg, chunks=1)
    path = ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    for f in range(cfg.past_frames):
        path.merge(dev(d.past_k[f], cfg.dtype), dev(d.past_v[f], cfg.dtype), f, F=1)
    torch.cuda.synchronize()
    return d, path


def _run(cfg, S, reuse=False):
    d, path = _setup(cfg)
    rep = Report()
    kp, vp = dev(d.prompt_k, cfg.dtype), dev(d.prompt_v, cfg.dtype)
    steps = denoise_steps(cfg, d, S)
    dense = O.denoise_schedule(S)
    first = cfg.past_frames
    pc, _ = O.hash_codes(d.prompt_k, d.planes, cfg.T, cfg.B)
    kept = None  # with reuse: the GPU's codes and kept lists of the first sparse step
    for s, (q, k, v) in enumerate(steps):
        st = cache_to_oracle(path.cache, cfg.dtype)
        path.denoise_step(s, S, dev(q, cfg.dtype), dev(k, cfg.dtype), dev(v, cfg.dtype), kp, vp, first,
                          reuse=reuse)
        torch.cuda.synchronize()
        assert int(path.status.item()) == 0
        if dense[s]:
            idx = np.tile(np.arange(cfg.P), (cfg.H, cfg.F, 1))
            cnt = np.full((cfg.H, cfg.F), cfg.P)
            qc = None
        elif kept is not None:
            # reused: the first sparse step's codes and kept lists, untouched
            qc, kc_first, idx, cnt = kept
            np.testing.assert_array_equal(host(path.q_codes).astype(np.uint32), qc)
            np.testing.assert_array_equal(host(path.kept_cnt), cnt)
            np.testing.assert_array_equal(host(path.kept_idx), idx)
        else:
            qc = check_codes(path.q_codes, q, d.planes, cfg.T, cfg.B, rep, f"step {s} query codes")
            gpc = host(path.p_codes[:, :, :cfg.P]).astype(np.uint32)
            assert not ((gpc ^ pc) & ~O.hash_codes(d.prompt_k, d.planes, cfg.T, cfg.B)[1]).any()
            idx, cnt = O.annca_prune(qc, gpc, cfg.F, cfg.n_f)
            np.testing.assert_array_equal(host(path.kept_cnt), cnt)
            np.testing.assert_array_equal(host(path.kept_idx), idx)
            if reuse:
                kept = (qc, host(path.k_codes).astype(np.uint32), idx, cnt)
        o_ca = O.annca_attention(q, d.prompt_k, d.prompt_v, idx, cnt, cfg.F, cfg.n_f, cfg.scale)
        check_att(path.o_ca, o_ca, f"step {s} cross", rep)
        if s + 1 < S:
            g = cache_to_oracle(path.cache, cfg.dtype)
            for name in ("K", "V", "m", "codes", "size"):
                np.testing.assert_array_equal(getattr(g, name), getattr(st, name), err_msg=f"step {s} wrote {name}")
            if dense[s]:
                kc = None
            elif reuse and s > _first_sparse(dense):
                kc = kept[1]  # the first sparse step's key codes, still in place
                np.testing.assert_array_equal(host(path.k_codes).astype(np.uint32), kc)
            else:
                kc = check_codes(path.k_codes, k, d.planes, cfg.T, cfg.B, rep, f"step {s} key codes")
            o_sa, lse = O.denoise_step_attention(q, qc, st, k, v, kc, dense[s], cfg.scale)
        else:
            kc = check_codes(path.k_codes, k, d.planes, cfg.T, cfg.B, rep, "last step key codes")
            st = check_merge(path, st, k, v, kc, path.match, cfg.F, cfg.n_f, first, cfg.tau, cfg.dtype, rep,
                             "last step merge")
            if dense[s]:
                view = O.CacheState(st.dtype, st.K, st.V, st.m, np.zeros((cfg.H, 1, cfg.C), np.uint32),
                                    st.last_frame, st.size, st.inserted, st.evicted)
                o_sa, lse = O.annsa_attention(q, np.zeros((cfg.H, 1, cfg.Nq), np.uint32), view, cfg.scale)
            else:
                o_sa, lse = O.annsa_attention(q, qc, st, cfg.scale)
        check_att(path.o_sa, o_sa, f"step {s} self", rep)
        gl = host(path.lse).astype(np.float64)
        fin = np.isfinite(lse)
        np.testing.assert_array_equal(np.isfinite(gl), fin)
        assert np.abs(gl[fin] - lse[fin]).max(initial=0) <= 1e-3
    return rep


def _first_sparse(dense):
    return dense.index(False) if False in dense else -1


def test_denoise_four_steps():
    """Steps 0 and 1 dense, step 2 sparse (cache + own keys), step 3 the
    merging chunk step (sparse): 2 heads, 300 tokens, 6 past frames."""
    cfg = CONFIGS[1].replace(H=2, n_f=300, F=1, past_frames=6, C=2048, P=64, redraw=0.3)
    _run(cfg, 4)


def test_denoise_single_dense_step_two_frames():
    """One step, hence dense and final: merge, then dense attention over the
    merged cache; two frames per chunk (per-frame cross-attention)."""
    cfg = CONFIGS[1].replace(H=2, n_f=200, F=2, past_frames=4, C=2048, P=48, redraw=0.3)
    _run(cfg, 1)


def test_denoise_reuse_codes_six_steps():
    """Codes computed once per chunk: steps 0 and 1 dense, steps 2 to 4
    sparse with the codes, query CSR and kept lists of step 2, step 5 the
    merging step (its keys hashed again, its queries' codes and kept lists
    still step 2's)."""
    cfg = CONFIGS[1].replace(H=2, n_f=300, F=1, past_frames=6, C=2048, P=64, redraw=0.3)
    _run(cfg, 6, reuse=True)
