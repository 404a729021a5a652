"""fastar_tempcache_merge_noalloc gives the same cache as fastar_tempcache_merge.

The no-allocation entry point is for callers that cannot allocate device
memory themselves, such as a plugin inside a host application that owns the
GPU's memory budget, or a C/FFI caller that only holds the pointers it was
given.  It takes its scratch from a fixed array inside the library instead
of a caller workspace.  Here two merge calls in a row run through both entry
points, via the C ABI, on two identical caches; every cache buffer and the
matches must agree bit for bit (both run the same kernels on the same
inputs, and the value update uses no atomics).  Before the compared calls a
merge of a larger problem runs through the no-allocation entry point on a
throwaway cache, so the shared array holds another problem's leftovers
when the compared calls read it.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import CONFIGS, layer_data

ERR_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE = 1, 2, 4


def _noalloc(L):
    import merged_attention_autoregressive_gb300 as fa
    f = L.fastar_tempcache_merge_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(fa.CacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int32, ctypes.c_float,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return f


def test_noalloc_rejects_problems_beyond_its_scratch():
    """40 heads x C 32768 x n_f 3600 needs about 56 MiB of scratch: refused, nothing launched."""
    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build
    build.build()
    f = _noalloc(fa.lib())
    fake = 0x1000
    cs = fa.CacheStruct(40, 128, 32768, 2, 10, 0, *([fake] * 10))
    rc = f(ctypes.byref(cs), fake, fake, fake, 3, 3600, 0, 0.95, None, None, None)
    assert rc == ERR_WORKSPACE
    # the one-layer workload (12 heads, C 32768, 1560 tokens per frame) fits
    assert fa.fastar_workspace_size(fa.OP_MERGE, 12, 1560, 128, 2, 8, 32768) <= 16 << 20


def test_noalloc_answers_like_the_workspace_merge():
    """Empty calls succeed and bad arguments are refused as the workspace
    merge refuses them, before any size check (no device is touched)."""
    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build
    build.build()
    f = _noalloc(fa.lib())
    fake = 0x1000
    cs = fa.CacheStruct(40, 128, 32768, 2, 10, 0, *([fake] * 10))
    for F, n_f in ((0, 3600), (3, 0)):
        assert f(ctypes.byref(cs), fake, fake, fake, F, n_f, 0, 0.95, None, None, None) == 0
    empty = fa.CacheStruct(0, 128, 32768, 2, 10, 0, *([fake] * 10))
    assert f(ctypes.byref(empty), fake, fake, fake, 3, 3600, 0, 0.95, None, None, None) == 0
    small = fa.CacheStruct(4, 128, 1024, 2, 8, 0, *([fake] * 10))
    assert f(ctypes.byref(small), fake, fake, fake, 3, 2048, 0, 0.95, None, None, None) == ERR_ARG
    big = fa.CacheStruct(1, 128, 8192, 2, 8, 0, *([fake] * 10))
    assert f(ctypes.byref(big), fake, fake, fake, 1, 7000, 0, 0.95, None, None, None) == ERR_UNSUPPORTED
    assert f(None, fake, fake, fake, 1, 10, 0, 0.95, None, None, None) == ERR_ARG


@pytest.mark.gpu
def test_noalloc_merge_matches_workspace_merge():
    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build
    build.build()
    f = _noalloc(fa.lib())
    cfg = CONFIGS[1].replace(H=4, n_f=300, F=2, past_frames=0, C=2048, redraw=0.3)
    d = layer_data(cfg, chunks=2)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.bfloat16)  # noqa: E731
    planes = bf(d.planes)
    A = fa.Cache(cfg.H, cfg.C, cfg.D, cfg.T, cfg.B)
    B = fa.Cache(cfg.H, cfg.C, cfg.D, cfg.T, cfg.B)
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # a larger merge (more heads, more keys per frame) through the shared
    # array first, on a throwaway cache: its leftovers must not matter
    big = cfg.replace(H=6, n_f=700, C=4096)
    dbig = layer_data(big, chunks=1)
    Z = fa.Cache(big.H, big.C, big.D, big.T, big.B)
    kz, vz = bf(dbig.chunk_k[0]), bf(dbig.chunk_v[0])
    cz = torch.empty(big.H, big.T, big.Nq, dtype=torch.int32, device="cuda")
    fa.fastar_hash(kz, bf(dbig.planes), big.T, big.B, cz, status=status[1:])
    for first in (0, big.F):
        zs = Z.struct()
        rc = f(ctypes.byref(zs), kz.data_ptr(), vz.data_ptr(), cz.data_ptr(), big.F, big.n_f, first,
               big.tau, None, status[1:].data_ptr(), stream)
        assert rc == 0, fa.STATUS.get(rc, rc)
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0]
    del Z
    for call in range(2):
        k, v = bf(d.chunk_k[call]), bf(d.chunk_v[call])
        codes = torch.empty(cfg.H, cfg.T, cfg.Nq, dtype=torch.int32, device="cuda")
        fa.fastar_hash(k, planes, cfg.T, cfg.B, codes, status=status[:1])
        match_a = torch.full((cfg.H, cfg.Nq), -7, dtype=torch.int32, device="cuda")
        match_b = torch.full((cfg.H, cfg.Nq), -7, dtype=torch.int32, device="cuda")
        first = call * cfg.F
        fa.fastar_tempcache_merge(A, k, v, codes, cfg.F, cfg.n_f, first, cfg.tau,
                                  match_out=match_a, status=status[:1])
        sb = B.struct()
        rc = f(ctypes.byref(sb), k.data_ptr(), v.data_ptr(), codes.data_ptr(), cfg.F, cfg.n_f,
               first, cfg.tau, match_b.data_ptr(), status[1:].data_ptr(), stream)
        assert rc == 0, fa.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0]
        assert torch.equal(match_a, match_b)
        assert (match_a >= -1).all()
        for name in ("K", "V", "m", "codes", "last_frame", "size", "inserted", "evicted"):
            assert torch.equal(getattr(A, name), getattr(B, name)), (call, name)
        n = A.size.tolist()
        for h in range(cfg.H):
            assert torch.equal(A.perm[h, :, :n[h]], B.perm[h, :, :n[h]])
        assert torch.equal(A.offsets, B.offsets)
    assert int(A.size.min()) > 0 and int((match_a >= 0).sum()) > 0
