"""fastar_tempcache_merge_noalloc gives the same cache as fastar_tempcache_merge.

The no-allocation entry point is for callers that cannot allocate device
memory themselves, such as a plugin inside a host application that owns the
GPU's memory budget, or a C/FFI caller that only holds the pointers it was
given.  It takes its scratch from a fixed array inside the library instead
of a caller workspace.  Here two merge calls in a row run through both entry
points, via the C ABI, on two identical caches; every cache buffer and the
matches must agree (integers exactly, values within one bf16 ulp, the
tolerance of the other merge tests).  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import CONFIGS, layer_data

ERR_WORKSPACE = 4


def _noalloc(L):
    import merged_attention_autoregressive_gb300 as fa
    f = L.fastar_tempcache_merge_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(fa.CacheStruct), ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int32, ctypes.c_float,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return f


def test_noalloc_rejects_problems_beyond_its_scratch():
    """40 heads x C 32768 x n_f 3600 needs about 55 MiB of scratch: refused, nothing launched."""
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
        for name in ("K", "m", "codes", "last_frame", "size", "inserted", "evicted"):
            assert torch.equal(getattr(A, name), getattr(B, name)), (call, name)
        va, vb = A.V.float(), B.V.float()
        ulp = torch.exp2(torch.floor(torch.log2(va.abs().clamp_min(2.0 ** -126))) - 7)
        assert ((va - vb).abs() <= ulp).all(), call
        n = A.size.tolist()
        for h in range(cfg.H):
            assert torch.equal(A.perm[h, :, :n[h]], B.perm[h, :, :n[h]])
        assert torch.equal(A.offsets, B.offsets)
    assert int(A.size.min()) > 0 and int((match_a >= 0).sum()) > 0
