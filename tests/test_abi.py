"""The C-ABI library builds for sm_103a, loads, and exports every declared call.

No compute is launched here: only calls that the host-side checks reject
(before any CUDA call) and the pure-host helpers are exercised, so these
tests run without a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fastar.h")


@pytest.fixture(scope="module")
def L():
    from merged_attention_autoregressive_gb300 import build, lib
    build.build()
    return lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fastar_\w+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("fastar_hash", "fastar_tempcache_merge", "fastar_annca_prune",
              "fastar_annca_attention", "fastar_annsa_attention", "fastar_workspace_size",
              "fastar_status_string", "fastar_version"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n
    assert L.fastar_version() >= 100


def test_binding_exports_match_header():
    import merged_attention_autoregressive_gb300 as m
    assert set(m.EXPORTS) <= set(declared_functions())


def test_status_strings(L):
    for code in (0, 1, 2, 3, 4, 16, 17, 18):
        assert L.fastar_status_string(code)
    assert L.fastar_status_string(12345) == b"unknown status"


def test_workspace_sizes(L):
    from merged_attention_autoregressive_gb300 import OP_HASH, OP_MERGE, OP_PRUNE
    assert L.fastar_workspace_size(OP_HASH, 12, 4680, 128, 2, 8, 32768) == 0
    assert L.fastar_workspace_size(OP_PRUNE, 12, 512, 128, 2, 8, 32768) == 0
    w1 = L.fastar_workspace_size(OP_MERGE, 12, 1560, 128, 2, 8, 32768)
    w2 = L.fastar_workspace_size(OP_MERGE, 24, 1560, 128, 2, 8, 32768)
    assert w1 >= 12 * 32768 * 16 and w2 >= 2 * w1 - 4096


def test_host_argument_errors_need_no_gpu(L):
    vp = ctypes.c_void_p
    fake = vp(0x1000)       # never dereferenced: the checks reject the call first
    # unsupported head dim
    assert L.fastar_hash(0, fake, 1, 8, 96, fake, 1, 4, fake, None, None, None, 0, None, None) == 2
    # T*B above 64
    assert L.fastar_hash(0, fake, 1, 8, 128, fake, 8, 9, fake, None, None, None, 0, None, None) == 2
    # perm without offsets
    assert L.fastar_hash(0, fake, 1, 8, 128, fake, 1, 4, fake, fake, None, None, 0, None, None) == 1
    # null input
    assert L.fastar_hash(0, None, 1, 8, 128, fake, 1, 4, fake, None, None, None, 0, None, None) == 1
    # misaligned rows
    assert L.fastar_hash(0, vp(0x1004), 1, 8, 128, fake, 1, 4, fake, None, None, None, 0, None,
                         None) == 1
    # empty input: nothing to do, OK without touching the device
    assert L.fastar_hash(0, None, 0, 8, 128, None, 1, 4, None, None, None, None, 0, None, None) == 0
    # prune: bad tables
    assert L.fastar_annca_prune(fake, fake, 1, 1, 4, 4, 0, 4, fake, fake, None, 0, None, None) == 1
    # attention: bad dtype
    assert L.fastar_annca_attention(7, fake, fake, fake, fake, fake, 1, 1, 4, 4, 128,
                                    ctypes.c_float(0.1), fake, None, 0, None, None) == 2
    # attention: scale must be positive and finite
    for bad in (0.0, -0.1, float("inf"), float("nan")):
        assert L.fastar_annca_attention(0, fake, fake, fake, fake, fake, 1, 1, 4, 4, 128,
                                        ctypes.c_float(bad), fake, None, 0, None, None) == 1
    # batched hash: job count, job arguments, head dim
    import merged_attention_autoregressive_gb300 as m
    jobs = (m.HashJob * 5)()
    for j in range(5):
        jobs[j] = m.HashJob(fake, 8, fake, None, None)
    L.fastar_hash_many.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(m.HashJob)] + \
        [ctypes.c_int] * 2 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                              ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]
    assert L.fastar_hash_many(0, 0, jobs, 1, 128, fake, 1, 4, None, 0, None, None) == 1
    assert L.fastar_hash_many(0, 5, jobs, 1, 128, fake, 1, 4, None, 0, None, None) == 1
    assert L.fastar_hash_many(0, 2, None, 1, 128, fake, 1, 4, None, 0, None, None) == 1
    assert L.fastar_hash_many(0, 2, jobs, 1, 96, fake, 1, 4, None, 0, None, None) == 2
    jobs[1] = m.HashJob(fake, 8, fake, fake, None)  # perm without offsets
    assert L.fastar_hash_many(0, 2, jobs, 1, 128, fake, 1, 4, None, 0, None, None) == 1
    jobs[1] = m.HashJob(vp(0x1004), 8, fake, None, None)  # misaligned rows
    assert L.fastar_hash_many(0, 2, jobs, 1, 128, fake, 1, 4, None, 0, None, None) == 1
    for j in range(2):
        jobs[j] = m.HashJob(None, 0, None, None, None)  # nothing to hash: OK, no device work
    assert L.fastar_hash_many(0, 2, jobs, 1, 128, None, 1, 4, None, 0, None, None) == 0
    # bucket CSR: sizes, bits, pointers
    L.fastar_bucket_csr.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert L.fastar_bucket_csr(fake, -1, 8, 4, fake, fake, None, None) == 1
    assert L.fastar_bucket_csr(fake, 2, 8, 13, fake, fake, None, None) == 2
    assert L.fastar_bucket_csr(None, 2, 8, 4, fake, fake, None, None) == 1
    assert L.fastar_bucket_csr(fake, 2, 8, 4, fake, None, None, None) == 1
    assert L.fastar_bucket_csr(None, 0, 8, 4, None, None, None, None) == 0
    # attention: the bf16 tensor-core path compacts the kept rows into ws
    assert L.fastar_annca_attention(0, fake, fake, fake, fake, fake, 1, 1, 4, 4, 128,
                                    ctypes.c_float(0.1), fake, None, 0, None, None) == 4
    need = L.fastar_workspace_size(3, 1, 1, 128, 0, 0, 4)
    assert need >= 2 * 64 * 128 * 2
    # merge with a codes-ready event: same argument checks
    assert L.fastar_tempcache_merge_ev(None, fake, fake, fake, 1, 4, 0, ctypes.c_float(0.9), None,
                                       None, 0, None, None, None) == 1
    # bounded-wait self-check: null status word, polls out of range
    L.fastar_check_bounded_wait.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    assert L.fastar_check_bounded_wait(8, None, None) == 1
    assert L.fastar_check_bounded_wait(0, fake, None) == 1
    assert L.fastar_check_bounded_wait(65537, fake, None) == 1
    # merge with a representative mode: unknown mode, mean-key without planes
    import merged_attention_autoregressive_gb300 as m2
    cs = m2.CacheStruct(1, 128, 64, 1, 4, 0, *([0x1000] * 10))
    for rep, planes in ((2, fake), (1, None), (1, vp(0x1004))):
        assert L.fastar_tempcache_merge_rep(ctypes.byref(cs), fake, fake, fake, 1, 4, 0, ctypes.c_float(0.9),
                                            rep, planes, None, None, 0, None, None, None) == 1
    # AnnSA partials / combine: slot range, head dim, workspace
    L.fastar_annsa_attention_part.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(m2.CacheStruct),
                                              ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]
    cs2 = m2.CacheStruct(1, 128, 64, 2, 4, 0, *([0x1000] * 10))
    for base, total in ((0, 5), (0, 0), (3, 4), (-1, 2)):   # T = 2 slots from base must fit in total <= 4
        assert L.fastar_annsa_attention_part(0, fake, fake, fake, fake, 8, ctypes.byref(cs2), ctypes.c_float(0.1),
                                             base, total, fake, 1 << 20, None, None) == 1
    assert L.fastar_annsa_attention_part(0, fake, fake, fake, fake, 8, ctypes.byref(cs2), ctypes.c_float(0.1),
                                         0, 2, fake, 16, None, None) == 4       # workspace too small
    L.fastar_annsa_combine.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_size_t] + [ctypes.c_void_p] * 4
    assert L.fastar_annsa_combine(1, 8, 128, 5, fake, 1 << 20, fake, None, None, None) == 1
    assert L.fastar_annsa_combine(1, 8, 64, 2, fake, 1 << 20, fake, None, None, None) == 2
    assert L.fastar_annsa_combine(1, 8, 128, 2, fake, 16, fake, None, None, None) == 4
    assert L.fastar_annsa_combine(0, 8, 128, 2, None, 0, None, None, None, None) == 0
    # merge: null cache
    assert L.fastar_tempcache_merge(None, fake, fake, fake, 1, 4, 0, ctypes.c_float(0.9), None,
                                    None, 0, None, None) == 1
    # merge: a frame above the frame-key limit (6144) or above the capacity;
    # no frames: nothing to do, OK without device work
    big = m2.CacheStruct(1, 128, 8192, 1, 4, 0, *([0x1000] * 10))
    assert L.fastar_tempcache_merge(ctypes.byref(big), fake, fake, fake, 1, 6145, 0, ctypes.c_float(0.9),
                                    None, None, 0, None, None) == 2
    assert L.fastar_tempcache_merge(ctypes.byref(cs), fake, fake, fake, 1, 65, 0, ctypes.c_float(0.9),
                                    None, None, 0, None, None) == 1
    assert L.fastar_tempcache_merge(ctypes.byref(cs), fake, fake, fake, 0, 4, 0, ctypes.c_float(0.9),
                                    None, None, 0, None, None) == 0


def test_annsa_parts_workspace_grows_with_slots(L):
    from merged_attention_autoregressive_gb300 import OP_ANNSA, OP_ANNSA_PARTS
    w1 = L.fastar_workspace_size(OP_ANNSA_PARTS, 12, 4680, 128, 1, 8, 32768)
    w4 = L.fastar_workspace_size(OP_ANNSA_PARTS, 12, 4680, 128, 4, 8, 32768)
    assert w1 >= 12 * 4680 * (128 * 2 + 8) and w4 >= 4 * 12 * 4680 * (128 * 2 + 8)
    # two slots hold what the two-table call keeps; a single table keeps nothing
    assert L.fastar_workspace_size(OP_ANNSA_PARTS, 12, 4680, 128, 2, 8, 32768) == \
        L.fastar_workspace_size(OP_ANNSA, 12, 4680, 128, 2, 8, 32768)
    assert L.fastar_workspace_size(OP_ANNSA, 12, 4680, 128, 1, 8, 32768) == 0
    assert L.fastar_workspace_size(OP_ANNSA_PARTS, 12, 4680, 128, 5, 8, 32768) == 0


def test_cache_view_describes_given_tensors():
    """Cache.view wraps existing tensors (here on the CPU: no device call)."""
    import torch
    import merged_attention_autoregressive_gb300 as m
    H, C, D, T, B = 2, 10, 128, 2, 3
    bufs = dict(K=torch.zeros(H, C, D, dtype=torch.bfloat16), V=torch.zeros(H, C, D, dtype=torch.bfloat16),
                m=torch.ones(H, C, dtype=torch.int32), codes=torch.zeros(H, T, C, dtype=torch.int32),
                last_frame=torch.zeros(H, C, dtype=torch.int32), size=torch.full((H,), C, dtype=torch.int32),
                inserted=torch.zeros(H, dtype=torch.int64), evicted=torch.zeros(H, dtype=torch.int64),
                perm=torch.zeros(H, T, C, dtype=torch.int32),
                offsets=torch.zeros(H, T, (1 << B) + 1, dtype=torch.int32))
    c = m.Cache.view(T, B, **bufs)
    assert (c.H, c.C, c.D, c.T, c.B) == (H, C, D, T, B)
    cs = c.struct()
    assert cs.K == bufs["K"].data_ptr() and cs.offsets == bufs["offsets"].data_ptr()
    assert (cs.H, cs.D, cs.C, cs.T, cs.B, cs.dt) == (H, D, C, T, B, m.BF16)


def test_merge_rejects_small_workspace(L):
    import merged_attention_autoregressive_gb300 as m
    fake = 0x1000
    cs = m.CacheStruct(2, 128, 64, 2, 8, 0, *([fake] * 10))
    rc = L.fastar_tempcache_merge(ctypes.byref(cs), ctypes.c_void_p(fake), ctypes.c_void_p(fake),
                                  ctypes.c_void_p(fake), 1, 16, 0, ctypes.c_float(0.9), None,
                                  ctypes.c_void_p(4096), 16, None, None)
    assert rc == 4
    # n_f above the capacity
    rc = L.fastar_tempcache_merge(ctypes.byref(cs), ctypes.c_void_p(fake), ctypes.c_void_p(fake),
                                  ctypes.c_void_p(fake), 1, 65, 0, ctypes.c_float(0.9), None,
                                  ctypes.c_void_p(4096), 1 << 30, None, None)
    assert rc == 1


def test_cache_checkpoint_round_trip(tmp_path):
    """Cache.save / Cache.load restore every buffer exactly (CPU tensors);
    a checkpoint of another shape is refused."""
    import torch
    import merged_attention_autoregressive_gb300 as m
    g = torch.Generator().manual_seed(3)
    a = m.Cache(2, 16, 64, 2, 3, torch.bfloat16, device="cpu")
    for n in a.BUFFERS:
        t = getattr(a, n)
        if t.is_floating_point():
            t.copy_(torch.randn(t.shape, generator=g).to(t.dtype))
        else:
            t.copy_(torch.randint(-5, 100, t.shape, generator=g).to(t.dtype))
    path = str(tmp_path / "cache.pt")
    a.save(path)
    b = m.Cache(2, 16, 64, 2, 3, torch.bfloat16, device="cpu")
    b.load(path)
    for n in a.BUFFERS:
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    c = m.Cache(2, 32, 64, 2, 3, torch.bfloat16, device="cpu")
    with pytest.raises(ValueError):
        c.load(path)
