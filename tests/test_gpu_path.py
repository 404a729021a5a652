"""GPU parity of the whole per-chunk path against the fp64 oracle (cascaded).

Runs the library through its C ABI (via the ctypes binding) on seeded
synthetic layers: the past frames are merged call by call, then one chunk
runs hash -> merge -> prune -> AnnCA -> AnnSA.  Every stage is compared with
the oracle as described in tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle as O
from parity import Report, cache_to_oracle, check_att, check_codes, check_csr, check_merge, dev, host
from workloads import CONFIGS, layer_data

pytestmark = pytest.mark.gpu


def _path(cfg, search="prev"):
    from merged_attention_autoregressive_gb300.path import ChunkPath
    return ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau,
                     dtype={"bf16": torch.bfloat16, "f32": torch.float32}[cfg.dtype], search=search)


def build_cache(cfg, d, path, rep, check=True):
    """Merge the past frames in calls of cfg.F frames; returns the oracle state."""
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    f = 0
    while f < cfg.past_frames:
        nF = min(cfg.F, cfg.past_frames - f)
        k = np.concatenate(d.past_k[f:f + nF], axis=1)
        v = np.concatenate(d.past_v[f:f + nF], axis=1)
        codes, match = path.merge(dev(k, cfg.dtype), dev(v, cfg.dtype), f, F=nF)
        torch.cuda.synchronize()
        if check:
            gc = check_codes(codes, k, d.planes, cfg.T, cfg.B, rep, f"past {f} key codes")
            st = check_merge(path, st, k, v, gc, match, nF, cfg.n_f, f, cfg.tau, cfg.dtype, rep,
                             f"past frames {f}..{f + nF - 1}", search=path.search)
            check_csr(path.cache.perm, path.cache.offsets, st.codes, 1 << cfg.B, st.size,
                      f"cache CSR after frame {f + nF - 1}")
        f += nF
    return st if check else cache_to_oracle(path.cache, cfg.dtype)


def run_chunk(cfg, d, path, st, rep, chunk=0, rows=None):
    q, k, v = d.chunk_q[chunk], d.chunk_k[chunk], d.chunk_v[chunk]
    first = cfg.past_frames + chunk * cfg.F
    qd, kd, vd = dev(q, cfg.dtype), dev(k, cfg.dtype), dev(v, cfg.dtype)
    kp, vp = dev(d.prompt_k, cfg.dtype), dev(d.prompt_v, cfg.dtype)
    path.step(qd, kd, vd, kp, vp, first)
    torch.cuda.synchronize()
    assert int(path.status.item()) == 0
    qc = check_codes(path.q_codes, q, d.planes, cfg.T, cfg.B, rep, "query codes")
    check_csr(path.q_perm, path.q_offsets, qc, 1 << cfg.B, what="query CSR")
    kc = check_codes(path.k_codes, k, d.planes, cfg.T, cfg.B, rep, "new key codes")
    pc = check_codes(path.p_codes[:, :, :cfg.P], d.prompt_k, d.planes, cfg.T, cfg.B, rep,
                     "prompt codes")
    st = check_merge(path, st, k, v, kc, path.match, cfg.F, cfg.n_f, first, cfg.tau, cfg.dtype,
                     rep, "chunk merge", search=path.search)
    check_csr(path.cache.perm, path.cache.offsets, st.codes, 1 << cfg.B, st.size, "cache CSR")
    idx, cnt = O.annca_prune(qc, pc, cfg.F, cfg.n_f)
    np.testing.assert_array_equal(host(path.kept_cnt), cnt)
    np.testing.assert_array_equal(host(path.kept_idx), idx)
    o_ca = O.annca_attention(q, d.prompt_k, d.prompt_v, idx, cnt, cfg.F, cfg.n_f, cfg.scale,
                             rows=rows)
    o_sa, lse = O.annsa_attention(q, qc, st, cfg.scale, rows=rows)
    sel = slice(None) if rows is None else rows
    check_att(path.o_ca[:, sel], o_ca, "AnnCA", rep)
    check_att(path.o_sa[:, sel], o_sa, "AnnSA", rep)
    gl = host(path.lse[:, sel]).astype(np.float64)
    fin = np.isfinite(lse)
    np.testing.assert_array_equal(np.isfinite(gl), fin)
    assert np.abs(gl[fin] - lse[fin]).max(initial=0) <= 1e-3
    return st


@pytest.mark.parametrize("C", [1024, 300])
def test_tiny_fp32_chain(C):
    """4 past frames + one 256-token frame, fp32; C = 300 forces eviction."""
    cfg = CONFIGS[0].replace(C=C)
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)
    if C == 300:
        assert int(host(path.cache.evicted).sum()) > 0


def test_tiny_bf16_chain():
    cfg = CONFIGS[0].replace(dtype="bf16", C=300)
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)


def test_ragged_bf16_chain():
    """Sizes off every tile multiple: n_f = 197, 2 frames, P = 77, T = 3, B = 7."""
    cfg = CONFIGS[0].replace(dtype="bf16", n_f=197, F=2, past_frames=5, P=77, T=3, B=7, C=700,
                             D=128, H=3, redraw=0.3)
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)


@pytest.mark.parametrize("tau", [1.5, -1.0])
def test_degenerate_thresholds_chain(tau):
    """The two degenerate thresholds on ragged sizes.  tau above 1: no key
    joins a group, so the cache is the append history of every key and
    evicts once full.  tau = -1: every key that has a candidate joins its
    best one, so nothing is inserted after the first frame and groups take
    several members in one frame (the merge's many-to-one path)."""
    cfg = CONFIGS[0].replace(dtype="bf16", n_f=197, F=2, past_frames=5, P=77, T=2, B=7, C=700,
                             D=128, H=2, redraw=0.3, tau=tau)
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)
    m = host(path.cache.m)
    match = host(path.match)
    if tau > 1:
        assert (match < 0).all() and int(m.max()) == 1
        assert int(host(path.cache.evicted).sum()) > 0
    else:
        assert (host(path.cache.size) == cfg.n_f).all()
        # some frame of the chunk has a slot that several of its keys joined
        per_frame = match.reshape(cfg.H, cfg.F, cfg.n_f)
        assert any(np.bincount(per_frame[h, f][per_frame[h, f] >= 0]).max() > 1
                   for h in range(cfg.H) for f in range(cfg.F))


def test_smaller_frames_after_larger_frames():
    """Calls of 300-key frames, then a call of 197-key frames on the same
    cache: the first frame of that call has more candidates (the ~300
    groups the previous frame refreshed) than keys, more than the staging
    copy holds, so the NN reads the candidates' scattered cache rows."""
    cfg = CONFIGS[0].replace(dtype="bf16", n_f=300, F=2, past_frames=4, P=77, T=2, B=7, C=2000,
                             D=128, H=3, redraw=0.3)
    d = layer_data(cfg)
    big = _path(cfg)
    big.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, big, rep)
    n_small = 197
    small = _path(cfg.replace(n_f=n_small))
    small.cache = big.cache
    small.planes.copy_(big.planes)
    first = cfg.past_frames
    assert int((np.asarray(st.last_frame) == first - 1).sum(axis=1).min()) > n_small
    cut = lambda a: np.concatenate([a[:, i * cfg.n_f:i * cfg.n_f + n_small] for i in range(cfg.F)], axis=1)  # noqa: E731
    k, v = cut(d.chunk_k[0]), cut(d.chunk_v[0])
    codes, match = small.merge(dev(k, cfg.dtype), dev(v, cfg.dtype), first, F=cfg.F)
    torch.cuda.synchronize()
    assert int(small.status.item()) == 0
    gc = check_codes(codes, k, d.planes, cfg.T, cfg.B, rep, "197-key frame codes")
    st = check_merge(small, st, k, v, gc, match, cfg.F, n_small, first, cfg.tau, cfg.dtype, rep,
                     "197-key frames after 300-key frames")
    check_csr(small.cache.perm, small.cache.offsets, st.codes, 1 << cfg.B, st.size, "cache CSR")
    assert int((host(match) >= 0).sum()) > 0


def test_largest_frame_and_bits():
    """The documented maxima: 6144 keys per frame (FASTAR_MAX_FRAME_KEYS),
    B = 12 (4096 buckets per table) with T * B = 48 hyperplanes, and a
    capacity the chunk's frame overflows, so the cache evicts."""
    cfg = CONFIGS[0].replace(dtype="bf16", n_f=6144, F=1, past_frames=2, P=64, T=4, B=12, C=8192,
                             D=128, H=2, redraw=0.3)
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)
    assert int(host(path.cache.evicted).min()) > 0


def test_wan_layer_chain():
    """Bench workload: 12 heads, D 128, 3 x 1560 queries, 21 merged past frames."""
    cfg = CONFIGS[1]
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)
    print("report", rep)


def test_long_prompt_prune_and_cross_attention():
    """4096-token prompt from 256 clusters, T = 4 x B = 10 (AnnCA stress)."""
    cfg = CONFIGS[3]
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    from merged_attention_autoregressive_gb300 import (fastar_annca_attention, fastar_annca_prune,
                                                       fastar_hash)
    q = d.chunk_q[0]
    qd, kp, vp = dev(q, cfg.dtype), dev(d.prompt_k, cfg.dtype), dev(d.prompt_v, cfg.dtype)
    fastar_hash(qd, path.planes, cfg.T, cfg.B, path.q_codes, status=path.status)
    fastar_hash(kp, path.planes, cfg.T, cfg.B, path.p_codes, status=path.status)
    fastar_annca_prune(path.q_codes, path.p_codes, cfg.F, cfg.n_f, cfg.B, path.kept_idx,
                       path.kept_cnt, status=path.status)
    fastar_annca_attention(qd, kp, vp, path.kept_idx, path.kept_cnt, cfg.F, cfg.n_f, cfg.scale,
                           path.o_ca, status=path.status)
    torch.cuda.synchronize()
    assert int(path.status.item()) == 0
    qc = check_codes(path.q_codes, q, d.planes, cfg.T, cfg.B, rep, "query codes")
    pc = check_codes(path.p_codes, d.prompt_k, d.planes, cfg.T, cfg.B, rep, "prompt codes")
    idx, cnt = O.annca_prune(qc, pc, cfg.F, cfg.n_f)
    np.testing.assert_array_equal(host(path.kept_cnt), cnt)
    np.testing.assert_array_equal(host(path.kept_idx), idx)
    ref = O.annca_attention(q, d.prompt_k, d.prompt_v, idx, cnt, cfg.F, cfg.n_f, cfg.scale)
    check_att(path.o_ca, ref, "AnnCA long prompt", rep)


def test_empty_sets_give_zero_output():
    """Empty kept sets and queries with no allowed slot give zeros (and lse -inf)."""
    cfg = CONFIGS[0].replace(dtype="bf16", H=2, D=128, n_f=64, F=2, past_frames=1, P=16, T=1, B=10)
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    from merged_attention_autoregressive_gb300 import (fastar_annca_attention, fastar_annca_prune,
                                                       fastar_annsa_attention)
    # crafted codes: prompt code 9 everywhere; queries code 5, except head 1 frame 1 (code 9)
    qc = torch.full((cfg.H, cfg.T, cfg.Nq), 5, dtype=torch.int32, device="cuda")
    pc = torch.full((cfg.H, cfg.T, cfg.P), 9, dtype=torch.int32, device="cuda")
    qc[1, :, cfg.n_f:] = 9
    fastar_annca_prune(qc, pc, cfg.F, cfg.n_f, cfg.B, path.kept_idx, path.kept_cnt,
                       status=path.status)
    q = dev(d.chunk_q[0], cfg.dtype)
    kp, vp = dev(d.prompt_k, cfg.dtype), dev(d.prompt_v, cfg.dtype)
    fastar_annca_attention(q, kp, vp, path.kept_idx, path.kept_cnt, cfg.F, cfg.n_f, cfg.scale,
                           path.o_ca, status=path.status)
    torch.cuda.synchronize()
    cnt = host(path.kept_cnt)
    assert cnt.tolist() == [[0, 0], [0, cfg.P]]
    o = host(path.o_ca)
    assert (o[0] == 0).all() and (o[1, :cfg.n_f] == 0).all()
    ref = O.annca_attention(d.chunk_q[0], d.prompt_k, d.prompt_v, host(path.kept_idx), cnt,
                            cfg.F, cfg.n_f, cfg.scale)
    check_att(path.o_ca, ref, "AnnCA crafted", rep)
    # AnnSA: half of the queries carry a code that no cache slot has
    used = set(st.codes[:, 0, :int(st.size.max())].ravel().tolist())
    absent = next(c for c in range(1 << cfg.B) if c not in used)
    qcodes = np.array(O.hash_codes(d.chunk_q[0], d.planes, cfg.T, cfg.B)[0])
    qcodes[:, :, ::2] = absent
    perm, offs = O.bucket_csr(qcodes, 1 << cfg.B)
    tq = lambda a: torch.from_numpy(np.ascontiguousarray(a).astype(np.int32)).cuda()  # noqa: E731
    fastar_annsa_attention(q, tq(qcodes), tq(perm), tq(offs), path.cache, cfg.scale, path.o_sa,
                           path.lse, ws=path.ws_annsa, status=path.status)
    torch.cuda.synchronize()
    assert int(path.status.item()) == 0
    o_sa, lse = O.annsa_attention(d.chunk_q[0], qcodes, st, cfg.scale)
    assert (host(path.o_sa)[:, ::2] == 0).all()
    assert np.isneginf(host(path.lse)[:, ::2]).all()
    check_att(path.o_sa, o_sa, "AnnSA crafted", rep)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_hash_many_equals_single_calls(dtype):
    """One batched hash pass gives exactly the codes and bucket CSR of one
    fastar_hash call per input (ragged row counts, an empty input, several
    128-row tiles and a partial last tile; bf16 uses the tensor-core kernel,
    fp32 the per-input fallback)."""
    from merged_attention_autoregressive_gb300 import fastar_hash, fastar_hash_many
    g = torch.Generator().manual_seed(7)
    H, D, T, B = 3, 128, 2, 8
    planes = torch.randn(T * B, D, generator=g).to(dtype).cuda()
    Ns = [517, 100, 0, 64]
    xs = [torch.randn(H, n, D, generator=g).to(dtype).cuda() for n in Ns]
    i32 = dict(dtype=torch.int32, device="cuda")
    many = [torch.full((H, T, max(n, 1)), -1, **i32) for n in Ns]
    perm = torch.full((H, T, Ns[0]), -1, **i32)
    offs = torch.full((H, T, (1 << B) + 1), -1, **i32)
    jobs = [(xs[0], many[0], perm, offs)] + [(xs[j], many[j][:, :, :Ns[j]], None, None)
                                             for j in range(1, len(Ns))]
    fastar_hash_many(jobs, planes, T, B)
    for j, n in enumerate(Ns):
        if n == 0:
            continue
        one = torch.full((H, T, n), -1, **i32)
        p1 = torch.full((H, T, n), -1, **i32) if j == 0 else None
        o1 = torch.full((H, T, (1 << B) + 1), -1, **i32) if j == 0 else None
        fastar_hash(xs[j], planes, T, B, one, p1, o1)
        torch.cuda.synchronize()
        assert torch.equal(many[j][:, :, :n].cpu(), one.cpu()), f"job {j} codes"
        if j == 0:
            assert torch.equal(perm.cpu(), p1.cpu()) and torch.equal(offs.cpu(), o1.cpu())


def test_step_host_matches_step():
    """The host-to-host chunk (inputs copied in per branch, outputs copied
    out as soon as they are final) gives exactly what the device chunk
    gives: same kernels, only the copies and the stream order differ."""
    cfg = CONFIGS[0].replace(dtype="bf16", n_f=197, F=2, past_frames=5, P=77, T=3, B=7, C=700,
                             D=128, H=3, redraw=0.3)
    d = layer_data(cfg)
    paths = [_path(cfg), _path(cfg)]
    for p in paths:
        p.planes.copy_(dev(d.planes, cfg.dtype))
        build_cache(cfg, d, p, Report(), check=False)
    a, b = paths
    ins = [dev(x, cfg.dtype) for x in (d.chunk_q[0], d.chunk_k[0], d.chunk_v[0], d.prompt_k, d.prompt_v)]
    first = cfg.past_frames
    a.step(*ins, first)
    hs = [x.cpu().pin_memory() for x in ins]
    ho_ca = torch.empty(b.o_ca.shape, dtype=b.o_ca.dtype).pin_memory()
    ho_sa = torch.empty(b.o_sa.shape, dtype=b.o_sa.dtype).pin_memory()
    b.step_host(*hs, ho_ca, ho_sa, first)
    torch.cuda.synchronize()
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    assert torch.equal(ho_ca, a.o_ca.cpu()) and torch.equal(ho_sa, a.o_sa.cpu())
    assert torch.equal(a.cache.K.cpu(), b.cache.K.cpu()) and torch.equal(a.match.cpu(), b.match.cpu())


def _sample_rows(nq, k, seed):
    return np.sort(np.random.default_rng(seed).choice(nq, size=min(k, nq), replace=False))


def test_14b_shapes_head_sample():
    """The 14B-like 720p layer's shapes (n_f 3600, Nq 10,800, 21 merged past
    frames, C 32,768, T 2 x B 10) on a seeded sample of layers and heads: heads are independent,
    so each sampled head's results equal its results inside the 40-head layer.
    Every index output is checked in full; attention on sampled query rows."""
    base = CONFIGS[4]
    for layer, heads in ((0, [0, 29]), (1, [13])):
        cfg = base.replace(H=len(heads))
        d = layer_data(cfg, layer=layer, chunks=1, heads=heads)
        path = _path(cfg)
        path.planes.copy_(dev(d.planes, cfg.dtype))
        rep = Report()
        st = build_cache(cfg, d, path, rep)
        run_chunk(cfg, d, path, st, rep, rows=_sample_rows(cfg.Nq, 192, layer))
        print("layer", layer, "heads", heads, "report", rep)


def test_rollout_head_sample():
    """The long-rollout workload's shapes (the one-layer Wan-1.3B-like chunk,
    5 % of keys redrawn per frame) from an empty cache,
    24 chunks on a seeded sample of heads, with the capacity cut to 4096 so
    that the cache fills (about chunk 12) and eviction runs from then on.
    Every chunk's indices and merge are checked against the oracle chain;
    attention on sampled rows of every chunk."""
    chunks = 24
    cfg = CONFIGS[2].replace(H=2, C=4096, chunks=chunks)
    d = layer_data(cfg, chunks=chunks, heads=[0, 11])
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    for c in range(chunks):
        st = run_chunk(cfg, d, path, st, rep, chunk=c,
                       rows=_sample_rows(cfg.Nq, 128 if c % 8 == 7 else 16, c))
    assert int(host(path.cache.size).min()) == cfg.C  # the cache filled up
    assert int(host(path.cache.evicted).sum()) > 0    # and evicted groups
    print("report", rep)


def test_recall_metrics_match_oracle():
    """The recall / density measurement of bench.py (the kernels' lse and
    kept lists against dense torch references) agrees with the oracle's
    definitions (retained softmax share, allowed density) on one chunk."""
    import bench
    cfg = CONFIGS[0].replace(dtype="bf16", n_f=197, F=2, past_frames=5, P=77, T=3, B=7, C=700,
                             D=128, H=3, redraw=0.3)
    d = layer_data(cfg)
    path = _path(cfg)
    path.planes.copy_(dev(d.planes, cfg.dtype))
    build_cache(cfg, d, path, Report(), check=False)
    ins = [dev(x, cfg.dtype) for x in (d.chunk_q[0], d.chunk_k[0], d.chunk_v[0], d.prompt_k, d.prompt_v)]
    path.step(*ins, cfg.past_frames)
    torch.cuda.synchronize()
    assert int(path.status.item()) == 0
    got = bench.recall_metrics(cfg, path, d, d.chunk_q[0])
    st = cache_to_oracle(path.cache, cfg.dtype)
    ret, dens = O.annsa_retained(d.chunk_q[0], host(path.q_codes), st, cfg.scale)
    assert abs(got["annsa_retained"] - ret.mean()) <= 2e-3 * ret.mean()
    assert abs(got["annsa_density"] - dens.mean()) <= 1e-6
    rca, share = O.annca_retained(d.chunk_q[0], d.prompt_k, host(path.kept_idx), host(path.kept_cnt),
                                  cfg.F, cfg.n_f, cfg.scale)
    assert abs(got["annca_retained"] - rca.mean()) <= 1e-4
    assert abs(got["annca_kept_share"] - share.mean()) <= 1e-6
