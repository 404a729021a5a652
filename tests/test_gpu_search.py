"""GPU parity of the TempCache search over every earlier frame.

The search variant (gist.science technical summary 2.A: the nearest earlier
key is looked for with LSH over the previous frames) matches each new key
against every live group that shares an LSH bucket with it, in any table,
instead of the previous frame's groups only.  Here it runs through the C ABI
(fastar_tempcache_merge_search via the chunk path) and is compared with the
oracle's tempcache_merge(search="lsh"), cascaded as in tests/parity.py:
NN decisions bit-exact outside listed near-ties, the cache state bit-exact
(V within one bf16 ulp), the CSRs, kept lists and attention as for the
method's search.  Workloads: the tiny fp32 chain with and without eviction,
a ragged bf16 chain (3 tables), and sampled heads of the Wan-1.3B-like layer
over several chunks with the capacity cut so that eviction runs.
"""
import numpy as np
import pytest

from parity import Report, dev, host
from test_gpu_path import _path, _sample_rows, build_cache, run_chunk
from workloads import CONFIGS, layer_data

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("C", [1024, 300])
def test_lsh_search_tiny_fp32(C):
    cfg = CONFIGS[0].replace(C=C, redraw=0.3)
    d = layer_data(cfg)
    path = _path(cfg, search="lsh")
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)
    if C == 300:
        assert int(host(path.cache.evicted).sum()) > 0


def test_lsh_search_ragged_bf16():
    cfg = CONFIGS[0].replace(dtype="bf16", n_f=197, F=2, past_frames=5, P=77, T=3, B=7, C=700,
                             D=128, H=3, redraw=0.3)
    d = layer_data(cfg)
    path = _path(cfg, search="lsh")
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    st = build_cache(cfg, d, path, rep)
    run_chunk(cfg, d, path, st, rep)


def test_lsh_search_wan_heads_with_eviction():
    """Two heads of the Wan-1.3B-like rollout shapes, 10 chunks from an empty
    cache cut to 4096 groups (it fills near chunk 6, then evicts).  From the
    fourth chunk on, 10 % of each frame's keys are replaced by copies (plus
    small noise) of groups that no frame has refreshed since before the
    previous frame, so that the search over every earlier frame has older
    groups to find; the keys are rounded to bf16 and given to both sides."""
    import oracle as O
    from workloads import round_bf16
    chunks = 10
    cfg = CONFIGS[2].replace(H=2, C=4096, chunks=chunks, redraw=0.2)
    d = layer_data(cfg, chunks=chunks, heads=[3, 7])
    path = _path(cfg, search="lsh")
    path.planes.copy_(dev(d.planes, cfg.dtype))
    rep = Report()
    rng = np.random.default_rng(11)
    st = O.CacheState.empty(cfg.H, cfg.C, cfg.D, cfg.T, cfg.dtype)
    older = 0
    for c in range(chunks):
        first = cfg.past_frames + c * cfg.F
        if c >= 3:
            k = d.chunk_k[c]
            for h in range(cfg.H):
                n = int(st.size[h])
                stale = np.nonzero(st.last_frame[h, :n] < first - 1)[0]
                for f in range(cfg.F):
                    pos = f * cfg.n_f + rng.choice(cfg.n_f, size=cfg.n_f // 10, replace=False)
                    src = rng.choice(stale, size=pos.size)
                    noisy = st.K[h, src] + 0.005 * rng.standard_normal((pos.size, cfg.D))
                    k[h, pos] = round_bf16(noisy.astype(np.float32))
        st_before = st
        st = run_chunk(cfg, d, path, st, rep, chunk=c, rows=_sample_rows(cfg.Nq, 64, c))
        m = host(path.match).astype(np.int64)
        # first frame of the chunk: matches to groups last refreshed before
        # the previous frame (the previous-frame search cannot make them)
        for h in range(cfg.H):
            for j in np.nonzero(m[h, :cfg.n_f] >= 0)[0]:
                older += int(st_before.last_frame[h, m[h, j]] < first - 1)
    assert int(host(path.cache.evicted).sum()) > 0
    assert older > 0, "no match reached an older frame's group"
    print("report", rep, "first-frame matches to older groups", older)
