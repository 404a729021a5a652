"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test fixes one function of the oracle to something independent of its
code: a fixture derived by hand from the pages' definitions
(tests/golden/*.txt), a closed form (Lemma 5.1 / A.1 of FAST-AR,
paperlayer.ai appendix A), a textbook law (random-hyperplane collision
probability 1 - theta/pi, Charikar 2002), a library routine computing the
same quantity by another route (scipy softmax / logsumexp, torch bf16
rounding), or an invariant of the definition.  A plausible mistake in the
oracle (a flipped bit order, a wrong sign of the log m bias, a missing
count, a wrong candidate frame, a strict instead of inclusive threshold,
dot products instead of cosines, a reversed eviction order) fails at least
one of them.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle as O
from golden_io import load


# ----------------------------------------------------------------- hashing
def test_hash_fixture_axis_planes():
    g = load("hash_axis_planes.txt")
    D, T, B = int(g["D"]), int(g["T"]), int(g["B"])
    R = np.stack([g[f"plane{i}"] for i in range(T * B)])
    x = np.stack([g[f"x{i}"] for i in range(4)])[None]
    codes, margin = O.hash_codes(x, R, T, B)
    assert codes.shape == (1, T, 4)
    np.testing.assert_array_equal(codes[0, 0], g["codes_t0"])
    np.testing.assert_array_equal(codes[0, 1], g["codes_t1"])
    np.testing.assert_array_equal(margin[0, 0], g["margin_t0"])
    np.testing.assert_array_equal(margin[0, 1], g["margin_t1"])


def test_hash_collision_law():
    """P[code_t(x) == code_t(y)] = (1 - theta/pi)^B for random hyperplanes."""
    rng = np.random.default_rng(7)
    D, B, T = 32, 3, 1
    n = 60000
    theta = 1.0
    x = rng.standard_normal((n, D))
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    u = rng.standard_normal((n, D))
    u -= (u * x).sum(1, keepdims=True) * x
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    y = math.cos(theta) * x + math.sin(theta) * u
    # one fresh hyperplane set per block of 100 pairs keeps the estimate unbiased
    hits = 0
    for blk in range(n // 100):
        R = rng.standard_normal((T * B, D))
        sl = slice(blk * 100, (blk + 1) * 100)
        cx, _ = O.hash_codes(x[None, sl], R, T, B)
        cy, _ = O.hash_codes(y[None, sl], R, T, B)
        hits += int((cx == cy).sum())
    p = hits / n
    expect = (1 - theta / math.pi) ** B
    sd = math.sqrt(expect * (1 - expect) / n)
    assert abs(p - expect) < 5 * sd + 0.01, (p, expect)


def test_hash_sign_and_scale_invariants():
    rng = np.random.default_rng(3)
    H, N, D, T, B = 2, 200, 16, 3, 5
    x = rng.standard_normal((H, N, D))
    R = rng.standard_normal((T * B, D))
    c, _ = O.hash_codes(x, R, T, B)
    c2, _ = O.hash_codes(3.5 * x, R, T, B)
    cn, _ = O.hash_codes(-x, R, T, B)
    np.testing.assert_array_equal(c, c2)
    np.testing.assert_array_equal(cn, (~c) & ((1 << B) - 1))
    assert c.max() < (1 << B)


def test_hash_margin_lists_near_zero_projections():
    R = np.array([[1.0, 0.0], [0.0, 1.0]])
    x = np.array([[[1.0, 1e-6], [1.0, 0.5]]])
    c, m = O.hash_codes(x, R, 1, 2)
    assert m[0, 0, 0] == 0b10 and m[0, 0, 1] == 0
    assert c[0, 0, 0] == 0b11 and c[0, 0, 1] == 0b11


# --------------------------------------------------------------------- CSR
def test_csr_fixture():
    g = load("csr_small.txt")
    perm, offs = O.bucket_csr(g["codes"], int(g["nbuckets"]))
    np.testing.assert_array_equal(perm, g["perm"])
    np.testing.assert_array_equal(offs, g["offsets"])
    perm, offs = O.bucket_csr(g["codes"], int(g["nbuckets"]), n=int(g["n_live"]))
    np.testing.assert_array_equal(perm, g["perm_live"])
    np.testing.assert_array_equal(offs, g["offsets_live"])


def test_csr_invariants_random():
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 64, size=(3, 2, 1000)).astype(np.uint32)
    perm, offs = O.bucket_csr(codes, 64)
    for g in range(3):
        for t in range(2):
            p, o, c = perm[g, t], offs[g, t], codes[g, t]
            assert sorted(p.tolist()) == list(range(1000))
            sc = c[p]
            assert np.all(np.diff(sc.astype(np.int64)) >= 0)
            for b in range(64):
                ids = p[o[b]:o[b + 1]]
                assert np.all(c[ids] == b)
                assert np.all(np.diff(ids) > 0)
            assert o[64] == 1000 and o[0] == 0


# ------------------------------------------------------------- round bf16
def test_round_storage_bf16_hand_values():
    # spacing of bf16 in [1, 2) is 2^-7
    cases = {1.0 + 2 ** -8: 1.0,                      # tie -> even (1.0)
             1.0 + 3 * 2 ** -8: 1.0 + 2 ** -6,        # tie -> even mantissa
             1.0 + 2 ** -8 + 2 ** -20: 1.0 + 2 ** -7,  # above the tie
             -(2.0 + 2 ** -7): -2.0,                  # spacing 2^-6, tie -> even
             3.0: 3.0, 0.0: 0.0}
    for x, want in cases.items():
        assert O.round_storage(np.array([x]), "bf16")[0] == want, x


def test_round_storage_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * rng.choice([1e-3, 1.0, 50.0], 20000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_storage(x.astype(np.float64), "bf16"), ref)


# --------------------------------------------------------------- TempCache
def _fixture_frames(g):
    frames = []
    for f in range(4):
        k = np.stack([g[f"f{f}_k0"], g[f"f{f}_k1"]])[None]
        v = np.stack([g[f"f{f}_v0"], g[f"f{f}_v1"]])[None]
        codes = np.asarray(g[f"f{f}_codes"], dtype=np.uint32).reshape(1, 1, 2)
        frames.append((k, v, codes, g[f"f{f}_match"]))
    return frames


def test_tempcache_fixture_frame_by_frame():
    g = load("tempcache_small.txt")
    st = O.CacheState.empty(1, int(g["C"]), int(g["D"]), 1, "f64")
    for f, (k, v, codes, want_match) in enumerate(_fixture_frames(g)):
        st, match, listed = O.tempcache_merge(st, k, v, codes, 1, 2, f, float(g["tau"]))
        np.testing.assert_array_equal(match[0], want_match)
        assert not listed.any()
    for s in range(3):
        np.testing.assert_array_equal(st.K[0, s], g[f"K{s}"])
        np.testing.assert_array_equal(st.V[0, s], g[f"V{s}"])
    np.testing.assert_array_equal(st.m[0], g["m"])
    np.testing.assert_array_equal(st.codes[0, 0], g["codes"])
    np.testing.assert_array_equal(st.last_frame[0], g["last_frame"])
    assert st.size[0] == g["size"] and st.inserted[0] == g["inserted"]
    assert st.evicted[0] == g["evicted"]


def test_tempcache_fixture_one_chunk_equals_frames():
    """Merging the four frames as one chunk gives the same state."""
    g = load("tempcache_small.txt")
    fr = _fixture_frames(g)
    k = np.concatenate([f[0] for f in fr], axis=1)
    v = np.concatenate([f[1] for f in fr], axis=1)
    c = np.concatenate([f[2] for f in fr], axis=2)
    st = O.CacheState.empty(1, 3, 4, 1, "f64")
    st, match, _ = O.tempcache_merge(st, k, v, c, 4, 2, 0, float(g["tau"]))
    np.testing.assert_array_equal(match[0], np.concatenate([f[3] for f in fr]))
    np.testing.assert_array_equal(st.m[0], g["m"])
    np.testing.assert_array_equal(st.V[0, 2], g["V2"])


def test_tempcache_eviction_ties_go_to_lowest_slot():
    g = load("tempcache_evict_ties.txt")
    st = O.CacheState.empty(1, 3, 6, 1, "f64")
    e = np.eye(6)
    z = lambda n: np.zeros((1, 1, n), np.uint32)  # noqa: E731
    where = lambda row: np.nonzero((st.K[0] == row).all(1))[0].tolist()  # noqa: E731
    st, _, _ = O.tempcache_merge(st, e[None, 0:3], np.ones((1, 3, 6)), z(3), 1, 3, 0, 0.9)
    st, m1, _ = O.tempcache_merge(st, e[None, 3:4], np.ones((1, 1, 6)), z(1), 1, 1, 1, 0.9)
    st, m2, _ = O.tempcache_merge(st, e[None, 4:6], np.ones((1, 2, 6)), z(2), 1, 2, 2, 0.9)
    assert (m1 == -1).all() and (m2 == -1).all()
    assert where(e[3]) == [g["slot_of_e3"]]
    assert where(e[4]) == [g["slot_of_e4"]]
    assert where(e[5]) == [g["slot_of_e5"]]
    np.testing.assert_array_equal(st.last_frame[0], g["last_frame"])
    assert st.evicted[0] == g["evicted"]


def test_tempcache_tie_goes_to_lowest_slot_and_threshold_inclusive():
    st = O.CacheState.empty(1, 8, 2, 1, "f64")
    # frame 0: two identical keys in slots 0 and 1, and (3,4) in slot 2
    k0 = np.array([[[1.0, 0.0], [1.0, 0.0], [3.0, 4.0]]])
    st, _, _ = O.tempcache_merge(st, k0, np.ones((1, 3, 2)), np.zeros((1, 1, 3), np.uint32),
                                 1, 3, 0, tau=2.0)          # tau > 1: no merging
    assert st.size[0] == 3
    # frame 1: (5,0) ties slots 0 and 1 at cos 1 -> slot 0;
    #          (0,1) has cos 4/5 = 0.8 with slot 2 -> matched at tau = 0.8
    k1 = np.array([[[5.0, 0.0], [0.0, 1.0]]])
    _, match, _ = O.tempcache_merge(st, k1, np.ones((1, 2, 2)), np.zeros((1, 1, 2), np.uint32),
                                    1, 2, 1, tau=0.8)
    np.testing.assert_array_equal(match[0], [0, 2])
    _, match, _ = O.tempcache_merge(st, k1, np.ones((1, 2, 2)), np.zeros((1, 1, 2), np.uint32),
                                    1, 2, 1, tau=0.8000001)
    np.testing.assert_array_equal(match[0], [0, -1])


def test_tempcache_uses_cosine_not_dot():
    st = O.CacheState.empty(1, 8, 2, 1, "f64")
    # slot 0 is long but off-direction, slot 1 short and aligned
    k0 = np.array([[[10.0, 10.0], [0.1, 0.0]]])
    st, _, _ = O.tempcache_merge(st, k0, np.ones((1, 2, 2)), np.zeros((1, 1, 2), np.uint32),
                                 1, 2, 0, tau=2.0)
    _, match, _ = O.tempcache_merge(st, np.array([[[1.0, 0.05]]]), np.ones((1, 1, 2)),
                                    np.zeros((1, 1, 1), np.uint32), 1, 1, 1, tau=0.9)
    assert match[0, 0] == 1


def test_tempcache_no_merge_above_one_is_append_history():
    rng = np.random.default_rng(2)
    H, n, D, F = 2, 5, 8, 3
    st = O.CacheState.empty(H, 64, D, 2, "f64")
    k = rng.standard_normal((H, F * n, D))
    v = rng.standard_normal((H, F * n, D))
    c = rng.integers(0, 8, size=(H, 2, F * n)).astype(np.uint32)
    st, match, _ = O.tempcache_merge(st, k, v, c, F, n, 10, tau=1.5)
    assert (match == -1).all()
    np.testing.assert_array_equal(st.K[:, :F * n], k)
    np.testing.assert_array_equal(st.V[:, :F * n], v)
    np.testing.assert_array_equal(st.last_frame[:, :F * n],
                                  np.repeat(np.arange(10, 10 + F), n)[None].repeat(H, 0))
    assert (st.m[:, :F * n] == 1).all() and (st.size == F * n).all()


def test_tempcache_lemma_end_to_end_closed_form():
    """Exact-permutation frames: the merged cache reproduces dense attention.

    Every new frame is an exact permutation of the previous one, so each key
    lineage stays one group (m = number of frames) whose value is the mean of
    its values.  By Lemma 5.1 attention over the merged cache with + ln m
    equals dense attention over the full unmerged history.
    """
    rng = np.random.default_rng(9)
    H, n, D, frames = 1, 12, 16, 5
    base = rng.standard_normal((n, D))
    st = O.CacheState.empty(H, 64, D, 1, "f64")
    allk, allv = [], []
    k = base
    for f in range(frames):
        if f:
            k = k[rng.permutation(n)]
        v = rng.standard_normal((n, D))
        allk.append(k)
        allv.append(v)
        st, match, _ = O.tempcache_merge(st, k[None], v[None], np.zeros((1, 1, n), np.uint32),
                                         1, n, f, tau=0.95)
    assert st.size[0] == n and (st.m[0, :n] == frames).all()
    q = rng.standard_normal((7, D))
    qc = np.zeros((1, 1, 7), np.uint32)
    o, lse = O.annsa_attention(q[None], qc, st, 1 / math.sqrt(D))
    K = np.concatenate(allk)
    V = np.concatenate(allv)
    s = (q @ K.T) / math.sqrt(D)
    ref = softmax(s, axis=1) @ V
    np.testing.assert_allclose(o[0], ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[0], logsumexp(s, axis=1), atol=1e-12, rtol=0)


def test_tempcache_invariants_on_synthetic_layer():
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[0].replace(C=300)            # small capacity: eviction happens
    d = layer_data(cfg)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    frames = d.past_k + [d.chunk_k[0]]
    values = d.past_v + [d.chunk_v[0]]
    inserted_keys = []
    for f, (k, v) in enumerate(zip(frames, values)):
        codes, _ = O.hash_codes(k, d.planes, cfg.T, cfg.B)
        st, match, listed = O.tempcache_merge(st, k, v, codes, 1, cfg.n_f, f, cfg.tau)
        inserted_keys.append(np.asarray(k[0], dtype=np.float64))
        assert st.m[0, :st.size[0]].sum() + st.evicted[0] == st.inserted[0]
        assert st.inserted[0] == (f + 1) * cfg.n_f
        assert (st.last_frame[0, :st.size[0]] <= f).all()
    assert st.evicted[0] > 0 and st.size[0] == cfg.C
    pool = {row.tobytes() for row in np.concatenate(inserted_keys)}
    assert all(st.K[0, s].tobytes() in pool for s in range(st.size[0]))
    codes, _ = O.hash_codes(st.K[:, :st.size[0]], d.planes, cfg.T, cfg.B)
    np.testing.assert_array_equal(codes, st.codes[:, :, :st.size[0]])


def _frames(g, nframes):
    out = []
    for f in range(nframes):
        k = np.stack([g[f"f{f}_k0"], g[f"f{f}_k1"]])[None]
        v = np.stack([g[f"f{f}_v0"], g[f"f{f}_v1"]])[None]
        codes = np.asarray(g[f"f{f}_codes"], dtype=np.uint32).reshape(1, 1, 2)
        out.append((k, v, codes, g[f"f{f}_match"]))
    return out


def test_tempcache_meankey_fixture():
    """Mean-key representative (paperlayer.ai appendix C) on a hand-derived
    history: the group key is the running count-weighted mean, its code the
    hash of that mean, and the next frame matches against it (a key that
    the mean accepts and the last key would not)."""
    g = load("tempcache_meankey_small.txt")
    D, C, tau = int(g["D"]), int(g["C"]), float(g["tau"])
    planes = np.asarray(g["planes"], dtype=np.float64).reshape(2, D)
    st = O.CacheState.empty(1, C, D, 1, "f64")
    for f, (k, v, codes, want) in enumerate(_frames(g, 3)):
        st, match, listed = O.tempcache_merge(st, k, v, codes, 1, 2, f, tau, rep="mean", planes=planes, B=2)
        np.testing.assert_array_equal(match[0], want)
        assert not listed.any()
    for s in range(3):
        np.testing.assert_array_equal(st.K[0, s], g[f"K{s}"])
        np.testing.assert_array_equal(st.V[0, s], g[f"V{s}"])
    np.testing.assert_array_equal(st.m[0], g["m"])
    np.testing.assert_array_equal(st.codes[0, 0], g["codes"])
    np.testing.assert_array_equal(st.last_frame[0], g["last_frame"])
    assert st.size[0] == g["size"] and st.inserted[0] == g["inserted"] and st.evicted[0] == g["evicted"]
    # the last-key mode keeps (1, 1/4) as the key of slot 0, which frame 2's
    # first key does not reach (cosine 0.8824): it opens a new group instead
    st = O.CacheState.empty(1, C, D, 1, "f64")
    for f, (k, v, codes, _) in enumerate(_frames(g, 3)):
        st, match, _ = O.tempcache_merge(st, k, v, codes, 1, 2, f, tau)
    np.testing.assert_array_equal(match[0], [-1, -1])
    np.testing.assert_array_equal(st.K[0, 0], [1, 0.25, 0, 0])
    assert st.size[0] == 4


def test_tempcache_meankey_equals_lastkey_on_exact_duplicates():
    """Closed form: the mean of identical keys is that key, so on frames that
    are exact permutations of each other the two representative modes give
    the same cache, bit for bit."""
    rng = np.random.default_rng(11)
    n, D, T, B = 10, 8, 2, 3
    planes = rng.standard_normal((T * B, D))
    base = rng.standard_normal((n, D))
    a = O.CacheState.empty(1, 32, D, T, "f64")
    b = O.CacheState.empty(1, 32, D, T, "f64")
    k = base
    for f in range(4):
        if f:
            k = k[rng.permutation(n)]
        v = rng.standard_normal((1, n, D))
        codes, _ = O.hash_codes(k[None], planes, T, B)
        a, ma, _ = O.tempcache_merge(a, k[None], v, codes, 1, n, f, 0.95)
        b, mb, _ = O.tempcache_merge(b, k[None], v, codes, 1, n, f, 0.95, rep="mean", planes=planes, B=B)
        np.testing.assert_array_equal(ma, mb)
    for name in ("K", "V", "m", "codes", "last_frame", "size", "inserted", "evicted"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name), err_msg=name)
    assert (a.m[0, :n] == 4).all()


def test_tempcache_meankey_invariants_on_synthetic_layer():
    """Mean-key mode on the tiny synthetic layer: every live group's codes
    are the hash of its stored key (outside margin bits), counts add up,
    and merged keys are means (not copies of an inserted key)."""
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[0].replace(C=300, redraw=0.3)
    d = layer_data(cfg)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    pool = set()
    for f, (k, v) in enumerate(zip(d.past_k + [d.chunk_k[0]], d.past_v + [d.chunk_v[0]])):
        codes, _ = O.hash_codes(k, d.planes, cfg.T, cfg.B)
        st, match, listed = O.tempcache_merge(st, k, v, codes, 1, cfg.n_f, f, cfg.tau, rep="mean",
                                              planes=d.planes, B=cfg.B)
        pool |= {row.tobytes() for row in np.asarray(k[0], dtype=np.float64)}
        assert st.m[0, :st.size[0]].sum() + st.evicted[0] == st.inserted[0]
    n = st.size[0]
    codes, margin = O.hash_codes(st.K[:, :n], d.planes, cfg.T, cfg.B)
    assert not ((codes ^ st.codes[:, :, :n]) & ~margin).any()
    merged = st.m[0, :n] > 1
    assert merged.any()
    assert sum(st.K[0, s].tobytes() not in pool for s in np.nonzero(merged)[0]) > 0


def test_tempcache_capacity_error():
    st = O.CacheState.empty(1, 2, 2, 1, "f64")
    k = np.array([[[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]])
    with pytest.raises(O.CapacityError):
        O.tempcache_merge(st, k, np.ones((1, 3, 2)), np.zeros((1, 1, 3), np.uint32), 1, 3, 0, 0.9)


# -------------------------------------------------------------------- AnnCA
def test_annca_prune_fixture():
    g = load("annca_prune_small.txt")
    F, n_f = int(g["F"]), int(g["n_f"])
    q = np.stack([g["q_t0"], g["q_t1"]])[None].astype(np.uint32)
    p = np.stack([g["p_t0"], g["p_t1"]])[None].astype(np.uint32)
    idx, cnt = O.annca_prune(q, p, F, n_f)
    np.testing.assert_array_equal(cnt[0], [3, 4])
    np.testing.assert_array_equal(idx[0, 0, :3], g["kept_f0"])
    np.testing.assert_array_equal(idx[0, 1, :4], g["kept_f1"])
    assert (idx[0, 0, 3:] == -1).all() and (idx[0, 1, 4:] == -1).all()


def test_annca_prune_bruteforce_invariant():
    rng = np.random.default_rng(4)
    H, T, F, n_f, P, nb = 2, 3, 2, 7, 40, 16
    q = rng.integers(0, nb, size=(H, T, F * n_f)).astype(np.uint32)
    p = rng.integers(0, nb, size=(H, T, P)).astype(np.uint32)
    idx, cnt = O.annca_prune(q, p, F, n_f)
    for h in range(H):
        for f in range(F):
            kept = set(idx[h, f, :cnt[h, f]].tolist())
            assert list(idx[h, f, :cnt[h, f]]) == sorted(kept)
            for j in range(P):
                shares = any(p[h, t, j] == q[h, t, f * n_f + i]
                             for t in range(T) for i in range(n_f))
                assert shares == (j in kept)


def test_annca_attention_matches_softmax_over_kept():
    rng = np.random.default_rng(8)
    H, F, n_f, P, D = 2, 2, 5, 9, 8
    q = rng.standard_normal((H, F * n_f, D))
    kp = rng.standard_normal((H, P, D))
    vp = rng.standard_normal((H, P, D))
    idx = np.full((H, F, P), -1, np.int32)
    cnt = np.zeros((H, F), np.int32)
    lists = {(0, 0): [1, 4, 7], (0, 1): [], (1, 0): list(range(P)), (1, 1): [0, 8]}
    for (h, f), ids in lists.items():
        idx[h, f, :len(ids)] = ids
        cnt[h, f] = len(ids)
    o = O.annca_attention(q, kp, vp, idx, cnt, F, n_f, 0.3)
    for (h, f), ids in lists.items():
        qs = q[h, f * n_f:(f + 1) * n_f]
        if not ids:
            assert (o[h, f * n_f:(f + 1) * n_f] == 0).all()
            continue
        ref = softmax(0.3 * qs @ kp[h, ids].T, axis=1) @ vp[h, ids]
        np.testing.assert_allclose(o[h, f * n_f:(f + 1) * n_f], ref, atol=1e-13, rtol=0)
    rows = np.array([9, 0, 6])
    o_rows = O.annca_attention(q, kp, vp, idx, cnt, F, n_f, 0.3, rows=rows)
    np.testing.assert_allclose(o_rows, o[:, rows], atol=1e-14, rtol=0)


# ---------------------------------------------------------- attention math
def test_lemma_5_1_merged_groups_equal_dense():
    """Lemma 5.1 / A.1: g groups of identical keys == g reps, mean V, + ln m."""
    rng = np.random.default_rng(1)
    D, g = 16, 6
    m = np.array([1, 3, 2, 7, 1, 4])
    reps = rng.standard_normal((g, D))
    K = np.repeat(reps, m, axis=0)
    V = rng.standard_normal((m.sum(), D))
    q = rng.standard_normal((5, D))
    ref = softmax(0.25 * q @ K.T, axis=1) @ V
    starts = np.concatenate([[0], np.cumsum(m)[:-1]])
    Vbar = np.stack([V[s:s + c].mean(0) for s, c in zip(starts, m)])
    o, lse = O.masked_attention(q, reps, Vbar, np.ones((5, g), bool), np.log(m), 0.25)
    np.testing.assert_allclose(o, ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, logsumexp(0.25 * q @ K.T, axis=1), atol=1e-12, rtol=0)
    # m_t = 1 everywhere: standard attention
    o1, _ = O.masked_attention(q, reps, Vbar, np.ones((5, g), bool), np.zeros(g), 0.25)
    np.testing.assert_allclose(o1, softmax(0.25 * q @ reps.T, axis=1) @ Vbar, atol=1e-12)


def test_masked_attention_equals_softmax_over_subset():
    rng = np.random.default_rng(12)
    n, M, D = 9, 30, 8
    q, k, v = (rng.standard_normal((n, D)), rng.standard_normal((M, D)),
               rng.standard_normal((M, D)))
    bias = rng.standard_normal(M)
    allowed = rng.random((n, M)) < 0.3
    allowed[3] = False
    o, lse = O.masked_attention(q, k, v, allowed, bias, 0.5)
    for i in range(n):
        ids = np.nonzero(allowed[i])[0]
        if ids.size == 0:
            assert (o[i] == 0).all() and lse[i] == -np.inf
            continue
        s = 0.5 * k[ids] @ q[i] + bias[ids]
        np.testing.assert_allclose(o[i], softmax(s) @ v[ids], atol=1e-13, rtol=0)
        np.testing.assert_allclose(lse[i], logsumexp(s), atol=1e-13)


def test_annsa_allowed_fixture_and_single_bucket_dense():
    g = load("annsa_allowed_small.txt")
    qc = np.stack([g["q_t0"], g["q_t1"]]).astype(np.uint32)
    kc = np.stack([g["k_t0"], g["k_t1"]]).astype(np.uint32)
    al = O.annsa_allowed(qc, kc)
    np.testing.assert_array_equal(al.astype(int), np.stack([g["allowed_q0"], g["allowed_q1"]]))
    # B = 0 special case: every code is 0, AnnSA reduces to dense attention
    rng = np.random.default_rng(13)
    H, C, D, n = 1, 16, 8, 6
    st = O.CacheState.empty(H, C, D, 2, "f64")
    st.K[0, :10] = rng.standard_normal((10, D))
    st.V[0, :10] = rng.standard_normal((10, D))
    st.m[0, :10] = rng.integers(1, 5, 10)
    st.size[0] = 10
    q = rng.standard_normal((1, n, D))
    o, lse = O.annsa_attention(q, np.zeros((1, 2, n), np.uint32), st, 0.35)
    s = 0.35 * q[0] @ st.K[0, :10].T + np.log(st.m[0, :10])
    np.testing.assert_allclose(o[0], softmax(s, axis=1) @ st.V[0, :10], atol=1e-13)
    np.testing.assert_allclose(lse[0], logsumexp(s, axis=1), atol=1e-13)


def test_retained_mass_is_the_allowed_softmax_share():
    """retained = exp(lse over the allowed keys - lse over all keys), an
    identity between two different computations (weights summed here,
    log-sum-exp in masked_attention), plus its end points."""
    rng = np.random.default_rng(11)
    n, M, D = 7, 19, 16
    q, k, v = rng.standard_normal((n, D)), rng.standard_normal((M, D)), rng.standard_normal((M, D))
    bias = np.log(rng.integers(1, 5, size=M).astype(np.float64))
    allowed = rng.random((n, M)) < 0.4
    allowed[:, 0] = True
    scale = 0.25
    r = O.retained_mass(q, k, allowed, bias, scale)
    _, lse_a = O.masked_attention(q, k, v, allowed, bias, scale)
    _, lse_all = O.masked_attention(q, k, v, np.ones((n, M), bool), bias, scale)
    np.testing.assert_allclose(r, np.exp(lse_a - lse_all), rtol=1e-12)
    np.testing.assert_allclose(r, [softmax(scale * q[i] @ k.T + bias)[allowed[i]].sum() for i in range(n)],
                               rtol=1e-12)
    np.testing.assert_array_equal(O.retained_mass(q, k, np.ones((n, M), bool), bias, scale), 1.0)
    np.testing.assert_array_equal(O.retained_mass(q, k, np.zeros((n, M), bool), bias, scale), 0.0)


def test_annsa_and_annca_retained_end_points():
    """One shared code everywhere: AnnSA keeps everything (retained 1,
    density 1); disjoint codes: nothing.  AnnCA with everything kept: 1."""
    rng = np.random.default_rng(12)
    H, T, D, Nq, C, size = 2, 2, 8, 5, 16, 9
    st = O.CacheState.empty(H, C, D, T, "f32")
    st.K[:, :size] = rng.standard_normal((H, size, D))
    st.m[:, :size] = rng.integers(1, 4, size=(H, size))
    st.size[:] = size
    q = rng.standard_normal((H, Nq, D))
    qc = np.zeros((H, T, Nq), np.uint32)
    st.codes[:] = 0
    r, dens = O.annsa_retained(q, qc, st, 0.3)
    np.testing.assert_allclose(r, 1.0, rtol=1e-12)
    np.testing.assert_array_equal(dens, 1.0)
    st.codes[:] = 1
    r, dens = O.annsa_retained(q, qc, st, 0.3)
    np.testing.assert_array_equal(r, 0.0)
    np.testing.assert_array_equal(dens, 0.0)
    P, F, n_f = 6, 1, Nq
    kp = rng.standard_normal((H, P, D))
    idx = np.tile(np.arange(P, dtype=np.int32), (H, F, 1))
    cnt = np.full((H, F), P, np.int32)
    r, share = O.annca_retained(q, kp, idx, cnt, F, n_f, 0.3)
    np.testing.assert_allclose(r, 1.0, rtol=1e-12)
    np.testing.assert_array_equal(share, 1.0)


# ------------------------------------------------------- denoising steps
def test_denoise_schedule_hand_values():
    """Sparse attention is off for the first 30 % of the denoising steps
    (paper.rainbus.top, limitations): step s is dense iff s < 0.3 S."""
    want = {1: [1], 2: [1, 0], 3: [1, 0, 0], 4: [1, 1, 0, 0], 5: [1, 1, 0, 0, 0],
            10: [1, 1, 1, 0, 0, 0, 0, 0, 0, 0]}
    for S, w in want.items():
        assert O.denoise_schedule(S) == [bool(x) for x in w], S


def _perm_history(rng, n, D, frames):
    st = O.CacheState.empty(1, 64, D, 1, "f64")
    allk, allv = [], []
    k = rng.standard_normal((n, D))
    for f in range(frames):
        if f:
            k = k[rng.permutation(n)]
        v = rng.standard_normal((n, D))
        allk.append(k)
        allv.append(v)
        st, _, _ = O.tempcache_merge(st, k[None], v[None], np.zeros((1, 1, n), np.uint32), 1, n, f, 0.95)
    return st, np.concatenate(allk), np.concatenate(allv)


def test_denoise_dense_step_equals_dense_attention_over_history_and_chunk():
    """A dense step over a cache of exact-duplicate groups equals dense
    softmax attention over the full unmerged history plus the step's own
    keys (Lemma 5.1 for the cache part; the step's keys count once)."""
    rng = np.random.default_rng(21)
    n, D = 10, 16
    st, Kh, Vh = _perm_history(rng, n, D, 4)
    q, k, v = (rng.standard_normal((1, 7, D)) for _ in range(3))
    codes = np.zeros((1, 1, 7), np.uint32)
    o, lse = O.denoise_step_attention(q, codes, st, k, v, codes, True, 1 / math.sqrt(D))
    K = np.concatenate([Kh, k[0]])
    V = np.concatenate([Vh, v[0]])
    s = (q[0] @ K.T) / math.sqrt(D)
    np.testing.assert_allclose(o[0], softmax(s, axis=1) @ V, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[0], logsumexp(s, axis=1), atol=1e-12, rtol=0)


def test_denoise_sparse_step_mask_by_brute_force():
    """A sparse step allows (query, key) iff some table's codes agree, on the
    cache's groups and on the step's own keys alike: checked against a mask
    built pair by pair and scipy's softmax over the allowed logits."""
    rng = np.random.default_rng(22)
    H, D, T, B, nq, nk, C = 1, 8, 2, 2, 6, 5, 16
    st = O.CacheState.empty(H, C, D, T, "f64")
    planes = rng.standard_normal((T * B, D))
    k0 = rng.standard_normal((1, 9, D))
    c0, _ = O.hash_codes(k0, planes, T, B)
    st, _, _ = O.tempcache_merge(st, k0, rng.standard_normal((1, 9, D)), c0, 1, 9, 0, 2.0)
    q, k, v = rng.standard_normal((1, nq, D)), rng.standard_normal((1, nk, D)), rng.standard_normal((1, nk, D))
    qc, _ = O.hash_codes(q, planes, T, B)
    kc, _ = O.hash_codes(k, planes, T, B)
    o, _ = O.denoise_step_attention(q, qc, st, k, v, kc, False, 0.5)
    size = int(st.size[0])
    keys = [st.K[0, s] for s in range(size)] + [k[0, j] for j in range(nk)]
    vals = [st.V[0, s] for s in range(size)] + [v[0, j] for j in range(nk)]
    kcodes = [[int(st.codes[0, t, s]) for t in range(T)] for s in range(size)] + \
        [[int(kc[0, t, j]) for t in range(T)] for j in range(nk)]
    for i in range(nq):
        ok = [any(int(qc[0, t, i]) == kcodes[j][t] for t in range(T)) for j in range(len(keys))]
        if not any(ok):
            np.testing.assert_array_equal(o[0, i], 0)
            continue
        logits = np.array([0.5 * q[0, i] @ keys[j] for j in range(len(keys)) if ok[j]])
        ref = softmax(logits) @ np.array([vals[j] for j in range(len(keys)) if ok[j]])
        np.testing.assert_allclose(o[0, i], ref, atol=1e-12, rtol=0)


def test_denoise_chunk_writes_the_cache_only_at_the_last_step():
    """Non-final steps leave the cache as it was; the final state is the
    TempCache merge of the last step's keys, and the last step attends the
    merged cache (dense when the schedule says so)."""
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[0].replace(redraw=0.3)
    d = layer_data(cfg)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    for f in range(cfg.past_frames):
        c, _ = O.hash_codes(d.past_k[f], d.planes, cfg.T, cfg.B)
        st, _, _ = O.tempcache_merge(st, d.past_k[f], d.past_v[f], c, 1, cfg.n_f, f, cfg.tau)
    rng = np.random.default_rng(5)
    steps = [tuple(x + rng.normal(0, 0.05 * (3 - s), x.shape) for x in (d.chunk_q[0], d.chunk_k[0], d.chunk_v[0]))
             for s in range(4)]
    before = st.copy()
    outs, fin, match = O.denoise_chunk(st, steps, d.prompt_k, d.prompt_v, d.planes, cfg.T, cfg.B, cfg.F,
                                       cfg.n_f, cfg.past_frames, cfg.tau, cfg.scale)
    for name in ("K", "V", "m", "codes", "size"):
        np.testing.assert_array_equal(getattr(st, name), getattr(before, name))
    kc, _ = O.hash_codes(steps[-1][1], d.planes, cfg.T, cfg.B)
    want, want_match, _ = O.tempcache_merge(before, steps[-1][1], steps[-1][2], kc, cfg.F, cfg.n_f,
                                            cfg.past_frames, cfg.tau)
    np.testing.assert_array_equal(fin.K, want.K)
    np.testing.assert_array_equal(match, want_match)
    qc, _ = O.hash_codes(steps[-1][0], d.planes, cfg.T, cfg.B)
    o_last, _ = O.annsa_attention(steps[-1][0], qc, fin, cfg.scale)   # step 3 of 4 is sparse
    np.testing.assert_array_equal(outs[-1][0], o_last)
    # a dense first step differs from its sparse counterpart (the schedule matters)
    q0, k0, v0 = steps[0]
    q0c, _ = O.hash_codes(q0, d.planes, cfg.T, cfg.B)
    k0c, _ = O.hash_codes(k0, d.planes, cfg.T, cfg.B)
    o_sparse, _ = O.denoise_step_attention(q0, q0c, before, k0, v0, k0c, False, cfg.scale)
    assert np.abs(outs[0][0] - o_sparse).max() > 1e-3


# ----------------------------------------------------- quantised ANN matcher
def test_quant_fixture_codes_and_top1():
    g = load("quant_small.txt")
    keys = np.asarray(g["keys"], dtype=np.float64).reshape(3, 2)
    lo, hi = O.sq_range(keys)
    np.testing.assert_array_equal(lo, g["lo"])
    np.testing.assert_array_equal(hi, g["hi"])
    np.testing.assert_array_equal(O.sq_encode(keys, lo, hi, 2).ravel(), g["codes_b2"])
    c1 = O.sq_encode(keys, lo, hi, 1)
    np.testing.assert_array_equal(c1.ravel(), g["codes_b1"])
    np.testing.assert_array_equal(O.sq_decode(c1, lo, hi, 1).ravel(), g["decoded_b1"])
    q = np.asarray(g["queries"], dtype=np.float64).reshape(3, 2)
    allowed = O.quant_topk(q, keys, np.zeros(3), 1, 1, 1.0)
    np.testing.assert_array_equal(np.argmax(allowed, axis=1), g["top1_b1"])
    assert (allowed.sum(axis=1) == 1).all()


def test_quant_error_bound_and_many_bits_equal_exact_topk():
    """|x - decode(encode(x))| <= step / 2 per coordinate; with 24 bits the
    quantised top-k is the exact top-k (random data, no near ties)."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((200, 16))
    lo, hi = O.sq_range(x)
    for bits in (2, 4, 8, 12):
        step = (hi - lo) / ((1 << bits) - 1)
        err = np.abs(O.sq_decode(O.sq_encode(x, lo, hi, bits), lo, hi, bits) - x)
        assert (err <= step / 2 + 1e-12).all(), bits
    q = rng.standard_normal((30, 16))
    bias = rng.standard_normal(200) * 0.1
    allowed = O.quant_topk(q, x, bias, 7, 24, 0.25)
    s = 0.25 * q @ x.T + bias
    srt = np.sort(s, axis=1)
    assert (srt[:, -7] - srt[:, -8] > 1e-6).all()
    exact = np.zeros_like(allowed)
    np.put_along_axis(exact, np.argsort(-s, axis=1)[:, :7], True, axis=1)
    np.testing.assert_array_equal(allowed, exact)


def test_quant_annsa_with_every_key_is_dense_attention():
    """k >= the live slots: the quantised matcher keeps everything and the
    output is the softmax over all logits scale q.K + ln m (scipy)."""
    rng = np.random.default_rng(32)
    H, D, n = 1, 8, 12
    st = O.CacheState.empty(H, 16, D, 1, "f64")
    st.K[0, :n] = rng.standard_normal((n, D))
    st.V[0, :n] = rng.standard_normal((n, D))
    st.m[0, :n] = rng.integers(1, 5, n)
    st.size[0] = n
    q = rng.standard_normal((1, 5, D))
    o, lse = O.annsa_quant_attention(q, st, 100, 4, 0.3)
    logits = 0.3 * q[0] @ st.K[0, :n].T + np.log(st.m[0, :n])
    np.testing.assert_allclose(o[0], softmax(logits, axis=1) @ st.V[0, :n], atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[0], logsumexp(logits, axis=1), atol=1e-12, rtol=0)
    # AnnCA likewise over every prompt token
    kp, vp = rng.standard_normal((1, 9, D)), rng.standard_normal((1, 9, D))
    oc = O.annca_quant_attention(q, kp, vp, 9, 2, 0.3)
    np.testing.assert_allclose(oc[0], softmax(0.3 * q[0] @ kp[0].T, axis=1) @ vp[0], atol=1e-12, rtol=0)


def test_quant_tempcache_matches_exact_at_many_bits_and_never_below_tau():
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[0].replace(redraw=0.3)
    d = layer_data(cfg)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    for f in range(cfg.past_frames):
        c, _ = O.hash_codes(d.past_k[f], d.planes, cfg.T, cfg.B)
        st, _, _ = O.tempcache_merge(st, d.past_k[f], d.past_v[f], c, 1, cfg.n_f, f, cfg.tau)
    k = d.chunk_k[0]
    f = cfg.past_frames
    exact, listed = O.tempcache_nn(st, k, f, cfg.tau)
    q24 = O.tempcache_nn_quant(st, k, f, cfg.tau, 24)
    np.testing.assert_array_equal(q24[~listed], exact[~listed])
    q1 = O.tempcache_nn_quant(st, k, f, cfg.tau, 1)
    kk = np.asarray(k[0], dtype=np.float64)
    for j in np.nonzero(q1[0] >= 0)[0]:
        s = q1[0, j]
        cos = kk[j] @ st.K[0, s] / (np.linalg.norm(kk[j]) * np.linalg.norm(st.K[0, s]))
        assert cos >= cfg.tau
    assert (q1[0] >= 0).sum() <= (exact[0] >= 0).sum() + listed.sum()


# ------------------------------------------ TempCache search over all previous frames
def test_tempcache_lsh_search_single_bucket_is_exact_search_over_all_groups():
    """With every code equal (one bucket) the LSH-candidate search is the
    exact top-1 cosine over every live group of earlier frames, checked by
    brute force; with the real codes a match always shares a bucket."""
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[0].replace(redraw=0.3)
    d = layer_data(cfg)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    for f in range(cfg.past_frames):
        c, _ = O.hash_codes(d.past_k[f], d.planes, cfg.T, cfg.B)
        st, _, _ = O.tempcache_merge(st, d.past_k[f], d.past_v[f], c, 1, cfg.n_f, f, cfg.tau)
    k = d.chunk_k[0]
    f = cfg.past_frames
    one = st.copy()
    one.codes[:] = 0
    match, listed = O.tempcache_nn_lsh(one, k, np.zeros((1, cfg.T, cfg.n_f), np.uint32), f, cfg.tau)
    kk = np.asarray(k[0], dtype=np.float64)
    size = int(st.size[0])
    for j in range(cfg.n_f):
        best, arg = -np.inf, -1
        for s in range(size):
            c = kk[j] @ st.K[0, s] / (np.linalg.norm(kk[j]) * np.linalg.norm(st.K[0, s]))
            if c > best:
                best, arg = c, s
        if listed[0, j]:
            continue
        assert match[0, j] == (arg if best >= cfg.tau else -1), j
    # the method's previous-frame search is a special case: every match it
    # makes among groups that share a bucket is found by the wider search too
    codes, _ = O.hash_codes(k, d.planes, cfg.T, cfg.B)
    wide, wl = O.tempcache_nn_lsh(st, k, codes, f, cfg.tau)
    for j in np.nonzero(wide[0] >= 0)[0]:
        s = wide[0, j]
        assert any(codes[0, t, j] == st.codes[0, t, s] for t in range(cfg.T))
    narrow, nl = O.tempcache_nn(st, k, f, cfg.tau)
    for j in np.nonzero(narrow[0] >= 0)[0]:
        s = narrow[0, j]
        shares = any(codes[0, t, j] == st.codes[0, t, s] for t in range(cfg.T))
        if shares and not (wl[0, j] or nl[0, j]):
            assert wide[0, j] >= 0, j   # that group is a candidate of the wider search too


def test_quant_topk_overlap_rises_with_precision():
    """The pages' precision ablation (paperlayer.ai appendix C: recall of
    the quantised matcher rises with the bits per value) on one synthetic
    head of the Wan-1.3B-like layer: the quantised top-k (k = 28 % of the
    live groups) shares more of the exact top-k as the bits grow, and all of
    it at 16 bits but for near-ties at the k-th score.  Measured here (400
    queries): 1 bit 0.876, 2 bits 0.898, 4 bits 0.977, 8 bits 0.9985,
    16 bits 0.999996."""
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[1].replace(H=1, past_frames=6)
    d = layer_data(cfg, chunks=1, heads=[0])
    st = O.CacheState.empty(1, cfg.C, cfg.D, cfg.T, cfg.dtype)
    for f in range(cfg.past_frames):
        c, _ = O.hash_codes(d.past_k[f], d.planes, cfg.T, cfg.B)
        st, _, _ = O.tempcache_merge(st, d.past_k[f], d.past_v[f], c, 1, cfg.n_f, f, cfg.tau)
    n = int(st.size[0])
    K, bias = st.K[0, :n], np.log(st.m[0, :n].astype(np.float64))
    q = np.asarray(d.chunk_q[0][0][:400], dtype=np.float64)
    k = int(0.28 * n)
    s = cfg.scale * q @ K.T + bias
    exact = np.zeros(s.shape, dtype=bool)
    np.put_along_axis(exact, np.argsort(-s, axis=1)[:, :k], True, axis=1)
    overlap = [float((O.quant_topk(q, K, bias, k, b, cfg.scale) & exact).sum() / exact.sum())
               for b in (1, 2, 4, 8, 16)]
    assert all(a <= b + 1e-12 for a, b in zip(overlap, overlap[1:])), overlap
    # at 16 bits only near-ties at the k-th score can swap a key
    assert overlap[0] < 0.95 and overlap[-1] >= 0.9999, overlap


# ------------------------------------------------ TempCache listing rule (hand cases)
# The near-boundary rule of the NN decision (an NN choice whose margin is
# below 1e-4 is listed and may go either way on the GPU): with tau = 0.95, a
# decision is listed iff its top-1 cosine lies within 1e-4 of tau, or its
# top-2 gap is below 1e-4 while the top-1 can still reach tau (top-1 >=
# tau - 1e-4).  Each case below puts unit key (1, 0) against candidates at
# hand-chosen cosines c, placed at (c, +-sqrt(1 - c^2)) (alternating sides)
# so that their cosine with the key is c to fp64 rounding; the expected
# match and listed flag follow from the rule by hand.
_TAU = 0.95
_NN_CASES = [
    # (candidate cosines in slot order, expected match slot, expected listed)
    ((1.0, 1.0), 0, True),                       # exact tie at cosine 1 -> lowest slot, listed
    ((_TAU + 5e-5,), 0, True),                   # top-1 just above tau: matched, listed
    ((_TAU - 5e-5,), -1, True),                  # top-1 just below tau: unmatched, listed
    ((_TAU - 0.01, _TAU - 0.01 + 5e-5), -1, False),   # near tie far below tau: not listed
    ((_TAU - 1.5e-4, _TAU - 2.0e-4), -1, False),  # near tie just beyond tau - 1e-4: not listed
    ((_TAU + 0.02, _TAU + 0.02 - 5e-5), 0, True),  # near tie above tau: listed, larger wins
    ((_TAU + 0.02 - 5e-5, _TAU + 0.02), 1, True),  # same, larger one in the higher slot
    ((_TAU + 0.02, _TAU + 0.02 - 2e-4), 0, False),  # gap 2e-4: a clear winner
    ((_TAU + 1.5e-4,), 0, False),                # 1.5e-4 above tau: outside the margin
    ((_TAU - 0.3, _TAU + 0.04, _TAU - 0.2), 1, False),  # clear winner in the middle slot
]


def _nn_state(cosines, frame=4, T=1):
    """Candidates at the given cosines to (1, 0), refreshed in frame-1, plus
    one live group of an older frame that is exactly aligned with the key
    (cosine 1) and must never be a candidate of the previous-frame search."""
    n = len(cosines)
    st = O.CacheState.empty(1, n + 4, 2, T, "f64")
    for s, c in enumerate(cosines):
        side = 1.0 if s % 2 == 0 else -1.0
        st.K[0, s] = (c, side * math.sqrt(max(0.0, 1.0 - c * c)))
        st.last_frame[0, s] = frame - 1
        st.m[0, s] = 1
    st.K[0, n] = (1.0, 0.0)
    st.last_frame[0, n] = frame - 2
    st.m[0, n] = 1
    st.size[0] = n + 1
    st.inserted[0] = n + 1
    return st


@pytest.mark.parametrize("cosines,want_match,want_listed", _NN_CASES)
def test_tempcache_nn_listing_rule_hand_cases(cosines, want_match, want_listed):
    st = _nn_state(cosines)
    k = np.array([[[1.0, 0.0]]])
    match, listed = O.tempcache_nn(st, k, 4, _TAU)
    assert match[0, 0] == want_match
    assert bool(listed[0, 0]) == want_listed


@pytest.mark.parametrize("cosines,want_match,want_listed", _NN_CASES)
def test_tempcache_nn_lsh_listing_rule_hand_cases(cosines, want_match, want_listed):
    """The search over every earlier frame lists by the same rule.  Every
    candidate shares the key's bucket here; the aligned older group is a
    candidate too, but it sits in another bucket, so it must be skipped:
    with it counted every case would match it at cosine 1."""
    st = _nn_state(cosines)
    n = len(cosines)
    st.codes[0, 0, :n] = 3
    st.codes[0, 0, n] = 5                      # the aligned older group: other bucket
    k = np.array([[[1.0, 0.0]]])
    match, listed = O.tempcache_nn_lsh(st, k, np.array([[[3]]], dtype=np.uint32), 4, _TAU)
    assert match[0, 0] == want_match
    assert bool(listed[0, 0]) == want_listed


def test_tempcache_nn_lsh_searches_older_frames_in_the_bucket():
    """An older group in the key's bucket is a candidate of the search over
    every earlier frame (not of the previous-frame search): put in the key's
    bucket, the aligned older group of the fixture wins at cosine 1, and an
    exact tie with it at cosine 1 is listed."""
    st = _nn_state((_TAU + 0.02,))
    st.codes[0, 0, :2] = 3
    k = np.array([[[1.0, 0.0]]])
    match, listed = O.tempcache_nn_lsh(st, k, np.array([[[3]]], dtype=np.uint32), 4, _TAU)
    assert match[0, 0] == 1 and not listed[0, 0]
    prev, _ = O.tempcache_nn(st, k, 4, _TAU)
    assert prev[0, 0] == 0
    st.K[0, 0] = (2.0, 0.0)                     # previous-frame group now aligned too
    match, listed = O.tempcache_nn_lsh(st, k, np.array([[[3]]], dtype=np.uint32), 4, _TAU)
    assert match[0, 0] == 0 and listed[0, 0]


def test_tempcache_merge_lsh_search_equals_previous_frame_search_after_one_frame():
    """After a single merged frame every live group was refreshed in that
    frame, so with every code equal (one bucket) the search over every
    earlier frame has exactly the previous-frame search's candidates: the
    next frame's merge must come out identical, bit for bit."""
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[0].replace(redraw=0.3)
    d = layer_data(cfg)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    zero = np.zeros((cfg.H, cfg.T, cfg.n_f), np.uint32)
    st, _, _ = O.tempcache_merge(st, d.past_k[0], d.past_v[0], zero, 1, cfg.n_f, 0, cfg.tau)
    a, ma, la = O.tempcache_merge(st, d.past_k[1], d.past_v[1], zero, 1, cfg.n_f, 1, cfg.tau)
    b, mb, lb = O.tempcache_merge(st, d.past_k[1], d.past_v[1], zero, 1, cfg.n_f, 1, cfg.tau, search="lsh")
    np.testing.assert_array_equal(ma, mb)
    np.testing.assert_array_equal(la, lb)
    assert (ma >= 0).any() and (ma < 0).any()
    for name in ("K", "V", "m", "codes", "last_frame", "size", "inserted", "evicted"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name), err_msg=name)


def test_tempcache_merge_lsh_search_reaches_older_groups_and_never_evicts_a_joined_one():
    """Hand history: frame 0 holds groups A = (1, 0) and B = (0, 1); frame 1
    only (0, 1) again (it joins B; A is not refreshed); in frame 2 the key
    (1, 0) finds A (refreshed in frame 0) with the search over every earlier
    frame but not with the previous-frame search; and with the capacity
    full, the evicted slot is an unmatched one, never the group just joined."""
    st = O.CacheState.empty(1, 3, 2, 1, "f64")
    z = lambda n: np.zeros((1, 1, n), np.uint32)  # noqa: E731
    st, _, _ = O.tempcache_merge(st, np.array([[[1.0, 0.0], [0.0, 1.0]]]), np.ones((1, 2, 2)), z(2), 1, 2, 0,
                                 0.95, search="lsh")
    st, m1, _ = O.tempcache_merge(st, np.array([[[0.0, 2.0]]]), np.ones((1, 1, 2)), z(1), 1, 1, 1, 0.95,
                                  search="lsh")
    assert m1[0].tolist() == [1]
    k2 = np.array([[[3.0, 0.0], [1.0, 1.0], [-1.0, 1.0]]])   # A, then two fresh keys
    lsh, m2, _ = O.tempcache_merge(st, k2, np.ones((1, 3, 2)), z(3), 1, 3, 2, 0.95, search="lsh")
    prev, m2p, _ = O.tempcache_merge(st, k2, np.ones((1, 3, 2)), z(3), 1, 3, 2, 0.95)
    assert m2[0].tolist() == [0, -1, -1]
    assert m2p[0].tolist() == [-1, -1, -1]
    # lsh: slot 2 is free (one insert), slot 1 (B, last refreshed in frame 1) is
    # evicted for the other; slot 0 (A, joined now) is kept
    assert lsh.last_frame[0].tolist() == [2, 2, 2] and lsh.m[0].tolist() == [2, 1, 1]
    assert lsh.evicted[0] == 2 and lsh.inserted[0] == 6


def test_quant_topk_listing_hand_cases():
    """Keys (0, 0), (1, 3), (3, 1) at 2 bits are decoded exactly (the hand
    fixture).  Query (1, 1) scores 0, 4, 4: with k = 1 the two keys at the
    boundary tie, so both are listed (either may be kept); query (1, 0)
    scores 0, 1, 3: with k = 1 key 2 is a clear winner, nothing is listed;
    with k = 3 (every key) nothing is listed either."""
    keys = np.array([[0.0, 0.0], [1.0, 3.0], [3.0, 1.0]])
    q = np.array([[1.0, 1.0], [1.0, 0.0]])
    allowed, listed = O.quant_topk_listed(q, keys, np.zeros(3), 1, 2, 1.0)
    assert allowed.tolist() == [[False, True, False], [False, False, True]]
    assert listed.tolist() == [[False, True, True], [False, False, False]]
    allowed, listed = O.quant_topk_listed(q, keys, np.zeros(3), 3, 2, 1.0)
    assert allowed.all() and not listed.any()
    # a bias that breaks the tie by more than the margin: nothing listed
    allowed, listed = O.quant_topk_listed(q, keys, np.array([0.0, 0.0, 0.01]), 1, 2, 1.0)
    assert allowed[0].tolist() == [False, False, True] and not listed[0].any()


def test_quant_tempcache_listing_hand_cases():
    """Candidates (1, 0) and (0, 1) (refreshed in frame 0) quantise exactly at
    any bits >= 1 (each coordinate is its range's end).  Key (1, 1) has
    approximate cosines 0.7071 to both: a tie, listed; its exact cosine is
    below tau = 0.95 anyway.  Key (1, 0.01) picks (1, 0) clearly, exact
    cosine 0.99995 >= tau: matched, not listed.  With tau = 0.99995 - 5e-5
    the same decision sits within the margin of tau: listed."""
    st = O.CacheState.empty(1, 4, 2, 1, "f64")
    st.K[0, :2] = [[1.0, 0.0], [0.0, 1.0]]
    st.last_frame[0, :2] = 0
    st.m[0, :2] = 1
    st.size[0] = 2
    k = np.array([[[1.0, 1.0], [1.0, 0.01]]])
    match, listed = O.tempcache_nn_quant_listed(st, k, 1, 0.95, 4)
    assert match[0].tolist() == [-1, 0]
    assert listed[0].tolist() == [True, False]
    c = 1.0 / math.sqrt(1.0 + 1e-4)
    match, listed = O.tempcache_nn_quant_listed(st, k, 1, c - 5e-5, 4)
    assert match[0].tolist() == [-1, 0] and listed[0].tolist() == [True, True]


def test_tempcache_merge_quant_search_at_many_bits_equals_the_exact_search():
    """At 20 bits the decoded candidates are the candidates to about 1e-6,
    so the quantised search's merge makes the exact search's decisions
    wherever neither is listed, and then the same cache."""
    from workloads import CONFIGS, layer_data
    cfg = CONFIGS[0].replace(redraw=0.3)
    d = layer_data(cfg)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    for f in range(cfg.past_frames):
        c, _ = O.hash_codes(d.past_k[f], d.planes, cfg.T, cfg.B)
        st, _, _ = O.tempcache_merge(st, d.past_k[f], d.past_v[f], c, 1, cfg.n_f, f, cfg.tau)
    c, _ = O.hash_codes(d.chunk_k[0], d.planes, cfg.T, cfg.B)
    a, ma, la = O.tempcache_merge(st, d.chunk_k[0], d.chunk_v[0], c, 1, cfg.n_f, cfg.past_frames, cfg.tau)
    b, mb, lb = O.tempcache_merge(st, d.chunk_k[0], d.chunk_v[0], c, 1, cfg.n_f, cfg.past_frames, cfg.tau,
                                  search="quant20")
    ok = ~(la | lb)
    np.testing.assert_array_equal(ma[ok], mb[ok])
    assert (ma >= 0).sum() > 10
    if (ma == mb).all():
        np.testing.assert_array_equal(a.K, b.K)
        np.testing.assert_array_equal(a.m, b.m)


def test_denoise_reuse_is_identity_when_the_steps_agree_and_reuses_otherwise():
    """With every step given the same inputs, reusing the first sparse
    step's codes and kept lists changes nothing (bit for bit); with the
    usual noisy steps the first sparse step is unchanged and a later sparse
    step attends with the first one's selection (checked against the plain
    step function given those codes)."""
    from workloads import CONFIGS, denoise_steps, layer_data
    cfg = CONFIGS[0].replace(F=1, n_f=64, past_frames=2, P=16, T=2, B=3)
    d = layer_data(cfg, chunks=1)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    for f in range(cfg.past_frames):
        c, _ = O.hash_codes(d.past_k[f], d.planes, cfg.T, cfg.B)
        st, _, _ = O.tempcache_merge(st, d.past_k[f], d.past_v[f], c, 1, cfg.n_f, f, cfg.tau)
    same = [(d.chunk_q[0], d.chunk_k[0], d.chunk_v[0])] * 5
    args = (d.prompt_k, d.prompt_v, d.planes, cfg.T, cfg.B, cfg.F, cfg.n_f, cfg.past_frames, cfg.tau, cfg.scale)
    a, sa, _ = O.denoise_chunk(st, same, *args)
    b, sb, _ = O.denoise_chunk(st, same, *args, reuse=True)
    for x, y in zip(a, b):
        for u, w in zip(x, y):
            np.testing.assert_array_equal(u, w)
    steps = denoise_steps(cfg, d, 5)
    a, _, _ = O.denoise_chunk(st, steps, *args)
    b, _, _ = O.denoise_chunk(st, steps, *args, reuse=True)
    dense = O.denoise_schedule(5)
    first = dense.index(False)
    np.testing.assert_array_equal(a[first][0], b[first][0])
    s = first + 1
    q, k, v = steps[s]
    q1, k1, _ = steps[first]
    qc, _ = O.hash_codes(q1, d.planes, cfg.T, cfg.B)
    kc, _ = O.hash_codes(k1, d.planes, cfg.T, cfg.B)
    o, lse = O.denoise_step_attention(q, qc, st, k, v, kc, False, cfg.scale)
    np.testing.assert_array_equal(b[s][0], o)
    assert not np.array_equal(a[s][0], b[s][0])
