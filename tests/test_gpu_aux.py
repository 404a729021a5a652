"""Failure detection, checkpoint / resume and determinism on the GPU.

* Failure detection without a fault: the library's bounded-wait error path
  is made to run out on purpose (a barrier that nothing arrives on, a few
  polls), and the test checks that the caller's status word reports it,
  that a later kernel given the same word writes nothing, and that the
  context still works.
* Checkpoint / resume: the cache is caller-owned device memory, so a
  checkpoint is a copy of its buffers.  A rollout that is snapshotted,
  continued, and then resumed from the snapshot in a second path (fresh
  workspaces and streams) must give bit-identical outputs and cache state:
  nothing the later chunks depend on lives outside the cache buffers, and
  the kernels are deterministic (atomics only pick maxima and minima,
  value sums run in a fixed order).
"""
import numpy as np
import pytest
import torch

from parity import Report, check_codes, dev
from workloads import CONFIGS, layer_data

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = 17
CACHE_BUFFERS = ("K", "V", "m", "codes", "last_frame", "size", "inserted", "evicted", "perm", "offsets")


def _path(cfg):
    from merged_attention_autoregressive_gb300.path import ChunkPath
    p = ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau)
    return p


def test_bounded_wait_timeout_is_reported_and_the_context_survives():
    import merged_attention_autoregressive_gb300 as fa
    cfg = CONFIGS[1].replace(H=2, n_f=300, F=1, past_frames=0, P=0)
    d = layer_data(cfg, chunks=1)
    x = dev(d.chunk_k[0], cfg.dtype)
    planes = dev(d.planes, cfg.dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fa.fastar_check_bounded_wait(64, status)
    torch.cuda.synchronize()
    assert int(status.item()) == ERR_TIMEOUT
    # the status word is sticky and every later kernel given it writes nothing
    codes = torch.full((cfg.H, cfg.T, cfg.Nq), -5, dtype=torch.int32, device="cuda")
    fa.fastar_hash(x, planes, cfg.T, cfg.B, codes, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ERR_TIMEOUT
    assert bool((codes == -5).all())
    # a second timeout does not overwrite the first error either
    fa.fastar_check_bounded_wait(1, status)
    torch.cuda.synchronize()
    assert int(status.item()) == ERR_TIMEOUT
    # the context is intact: the same call with a clean word is correct
    clean = torch.zeros(1, dtype=torch.int32, device="cuda")
    fa.fastar_hash(x, planes, cfg.T, cfg.B, codes, status=clean)
    torch.cuda.synchronize()
    assert int(clean.item()) == 0
    check_codes(codes, d.chunk_k[0], d.planes, cfg.T, cfg.B, Report(), "hash after a timeout")


def _chunks(path, d, cfg, start, stop):
    kp, vp = dev(d.prompt_k, cfg.dtype), dev(d.prompt_v, cfg.dtype)
    outs = []
    for c in range(start, stop):
        q, k, v = (dev(x[c], cfg.dtype) for x in (d.chunk_q, d.chunk_k, d.chunk_v))
        path.step(q, k, v, kp, vp, c * cfg.F)
        outs.append([t.clone() for t in (path.o_sa, path.o_ca, path.lse, path.match, path.kept_cnt)])
    torch.cuda.synchronize()
    assert int(path.status.item()) == 0
    return outs


def test_checkpoint_resume_is_bit_identical():
    """6 chunks of 2 frames x 300 keys into a 1024-slot cache (full, and
    evicting, in the last two chunks): snapshot after 3 chunks, run 3 more;
    a second path restored from the snapshot runs the same 3 chunks."""
    cfg = CONFIGS[1].replace(H=2, n_f=300, F=2, past_frames=0, C=1024, P=96, redraw=0.3)
    d = layer_data(cfg, chunks=6)
    a = _path(cfg)
    a.planes.copy_(dev(d.planes, cfg.dtype))
    _chunks(a, d, cfg, 0, 3)
    snap = {n: getattr(a.cache, n).clone() for n in CACHE_BUFFERS}
    ref = _chunks(a, d, cfg, 3, 6)
    assert int(a.cache.evicted.sum()) > 0, "the rollout should evict"
    b = _path(cfg)
    b.planes.copy_(dev(d.planes, cfg.dtype))
    for n in CACHE_BUFFERS:
        getattr(b.cache, n).copy_(snap[n])
    got = _chunks(b, d, cfg, 3, 6)
    for c, (r, g) in enumerate(zip(ref, got)):
        for name, x, y in zip(("o_sa", "o_ca", "lse", "match", "kept_cnt"), r, g):
            assert torch.equal(x, y), (c, name)
    for n in CACHE_BUFFERS:
        assert torch.equal(getattr(a.cache, n), getattr(b.cache, n)), n
    inserted = int(a.cache.inserted.sum())
    assert inserted == cfg.H * 6 * cfg.F * cfg.n_f
    # unused slots hold m = 0, so this holds whether or not the cache is full
    assert int(a.cache.m.long().sum()) + int(a.cache.evicted.sum()) == inserted
    assert np.isfinite(ref[-1][2].float().cpu().numpy()).any()


def test_one_bucket_cache_gives_dense_attention():
    """With every code 0 (one table, one bit) and m = 1 everywhere, AnnSA is
    plain softmax attention over every cached key, and AnnCA with every
    prompt token kept is plain cross-attention: both against the oracle's
    fp64 attention with everything allowed (the bench's dense run)."""
    import merged_attention_autoregressive_gb300 as fa
    import oracle as O
    rng = np.random.default_rng(7)
    H, n, Nq, P, F, D = 2, 700, 300, 90, 2, 128
    n_f = Nq // F
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to("cuda", torch.bfloat16)  # noqa: E731
    K, V, q = bf(rng.normal(size=(H, n, D))), bf(rng.normal(size=(H, n, D))), bf(rng.normal(size=(H, Nq, D)))
    kp, vp = bf(rng.normal(size=(H, P, D))), bf(rng.normal(size=(H, P, D)))
    i32 = dict(dtype=torch.int32, device="cuda")
    c = fa.Cache(H, n, D, 1, 1)
    c.K.copy_(K)
    c.V.copy_(V)
    c.m.fill_(1)
    c.last_frame.zero_()
    c.size.fill_(n)
    c.perm[:, 0].copy_(torch.arange(n, **i32))
    c.offsets[:, 0] = torch.tensor([0, n, n], **i32)
    q_codes = torch.zeros(H, 1, Nq, **i32)
    q_perm = torch.arange(Nq, **i32).repeat(H, 1, 1).contiguous()
    q_off = torch.tensor([0, Nq, Nq], **i32).repeat(H, 1, 1).contiguous()
    o_sa = torch.empty(H, Nq, D, dtype=torch.bfloat16, device="cuda")
    o_ca = torch.empty_like(o_sa)
    st = torch.zeros(1, **i32)
    scale = D ** -0.5
    fa.fastar_annsa_attention(q, q_codes, q_perm, q_off, c, scale, o_sa, status=st)
    kept_idx = torch.arange(P, **i32).repeat(H, F, 1).contiguous()
    kept_cnt = torch.full((H, F), P, **i32)
    fa.fastar_annca_attention(q, kp, vp, kept_idx, kept_cnt, F, n_f, scale, o_ca, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    h64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    for h in range(H):
        for out, kk, vv in ((o_sa, K, V), (o_ca, kp, vp)):
            ref = O.masked_attention(h64(q[h]), h64(kk[h]), h64(vv[h]),
                                     np.ones((Nq, kk.shape[1]), bool), np.zeros(kk.shape[1]), scale)
            ref = ref[0] if isinstance(ref, tuple) else ref
            err = np.abs(h64(out[h]) - ref)
            assert err.max() <= 1e-2 and err.mean() <= 1e-3, (h, err.max(), err.mean())
