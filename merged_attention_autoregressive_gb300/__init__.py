"""Python binding of libfastar, the FAST-AR per-chunk attention library.

Argument marshalling only: every function reads shapes from torch tensors,
passes their device pointers and the current CUDA stream to the C ABI of
include/fastar.h, and raises FastarError on a non-zero status.  All work
runs in the library's CUDA kernels; there is no fallback.  If the library
has not been built, loading it raises (build it with
`python -m merged_attention_autoregressive_gb300.build`).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfastar.so")

BF16, F32 = 0, 1
OP_HASH, OP_MERGE, OP_PRUNE, OP_ANNCA, OP_ANNSA, OP_ANNSA_PARTS = 0, 1, 2, 3, 4, 5
REP_LAST, REP_MEAN = 0, 1
REPS = {"last": REP_LAST, "mean": REP_MEAN}
SEARCH_PREV, SEARCH_LSH, SEARCH_QUANT = 0, 1, 2
OP_QUANT = 6


def search_code(search: str) -> int:
    """"prev", "lsh" or "quant<bits>" (e.g. "quant8") as the C ABI's search value."""
    if search == "prev":
        return SEARCH_PREV
    if search == "lsh":
        return SEARCH_LSH
    if search.startswith("quant"):
        bits = int(search[5:])
        return SEARCH_QUANT | (bits << 8)
    raise ValueError(f"unknown search {search!r}")
STATUS = {0: "FASTAR_OK", 1: "FASTAR_ERR_ARG", 2: "FASTAR_ERR_UNSUPPORTED", 3: "FASTAR_ERR_CUDA",
          4: "FASTAR_ERR_WORKSPACE", 16: "FASTAR_ERR_CAPACITY", 17: "FASTAR_ERR_TIMEOUT",
          18: "FASTAR_ERR_DEVICE_ARG"}
EXPORTS = ["fastar_status_string", "fastar_version", "fastar_launch_count",
           "fastar_timing_begin", "fastar_timing_end", "fastar_timing_name",
           "fastar_workspace_size", "fastar_hash", "fastar_hash_many", "fastar_bucket_csr",
           "fastar_tempcache_merge", "fastar_tempcache_merge_ev", "fastar_annca_prune", "fastar_annca_attention",
           "fastar_annsa_attention", "fastar_check_bounded_wait", "fastar_tempcache_merge_rep",
           "fastar_annsa_attention_part", "fastar_annsa_combine", "fastar_tempcache_merge_search",
           "fastar_annsa_quant_attention", "fastar_annca_quant_attention"]


class FastarError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)} ({lib().fastar_status_string(code).decode()})")
        self.code = code


class CacheStruct(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("D", ctypes.c_int), ("C", ctypes.c_int),
                ("T", ctypes.c_int), ("B", ctypes.c_int), ("dt", ctypes.c_int),
                ("K", ctypes.c_void_p), ("V", ctypes.c_void_p), ("m", ctypes.c_void_p),
                ("codes", ctypes.c_void_p), ("last_frame", ctypes.c_void_p),
                ("size", ctypes.c_void_p), ("inserted", ctypes.c_void_p),
                ("evicted", ctypes.c_void_p), ("perm", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p)]


_lib = None
_VP, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
MAX_HASH_JOBS = 4


class HashJob(ctypes.Structure):
    """fastar_hash_job: one input of fastar_hash_many."""
    _fields_ = [("x", _VP), ("N", _I), ("codes", _VP), ("perm", _VP), ("offsets", _VP)]


def lib() -> ctypes.CDLL:
    """Load the in-tree libfastar.so (raises OSError when it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with "
                          "`python -m merged_attention_autoregressive_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.fastar_status_string.restype = ctypes.c_char_p
        L.fastar_status_string.argtypes = [_I]
        L.fastar_version.restype = _I
        L.fastar_launch_count.restype = ctypes.c_uint64
        L.fastar_timing_begin.argtypes = [_VP, _I]
        L.fastar_timing_begin.restype = _I
        L.fastar_timing_end.restype = _I
        L.fastar_timing_name.argtypes = [_I]
        L.fastar_timing_name.restype = ctypes.c_char_p
        L.fastar_workspace_size.restype = _SZ
        L.fastar_workspace_size.argtypes = [_I] * 7
        L.fastar_hash.argtypes = [_I, _VP, _I, _I, _I, _VP, _I, _I, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]
        L.fastar_bucket_csr.argtypes = [_VP, _I, _I, _I, _VP, _VP, _VP, _VP]
        L.fastar_hash_many.argtypes = [_I, _I, ctypes.POINTER(HashJob), _I, _I, _VP, _I, _I, _VP, _SZ,
                                       _VP, _VP]
        L.fastar_tempcache_merge.argtypes = [ctypes.POINTER(CacheStruct), _VP, _VP, _VP, _I, _I,
                                             ctypes.c_int32, _F, _VP, _VP, _SZ, _VP, _VP]
        L.fastar_tempcache_merge_ev.argtypes = [ctypes.POINTER(CacheStruct), _VP, _VP, _VP, _I, _I,
                                                ctypes.c_int32, _F, _VP, _VP, _SZ, _VP, _VP, _VP]
        L.fastar_annca_prune.argtypes = [_VP, _VP, _I, _I, _I, _I, _I, _I, _VP, _VP, _VP, _SZ, _VP, _VP]
        L.fastar_annca_attention.argtypes = [_I, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F,
                                             _VP, _VP, _SZ, _VP, _VP]
        L.fastar_annsa_attention.argtypes = [_I, _VP, _VP, _VP, _VP, _I, ctypes.POINTER(CacheStruct),
                                             _F, _VP, _VP, _VP, _SZ, _VP, _VP]
        L.fastar_check_bounded_wait.argtypes = [_I, _VP, _VP]
        L.fastar_annsa_attention_part.argtypes = [_I, _VP, _VP, _VP, _VP, _I, ctypes.POINTER(CacheStruct),
                                                  _F, _I, _I, _VP, _SZ, _VP, _VP]
        L.fastar_annsa_combine.argtypes = [_I, _I, _I, _I, _VP, _SZ, _VP, _VP, _VP, _VP]
        L.fastar_tempcache_merge_rep.argtypes = [ctypes.POINTER(CacheStruct), _VP, _VP, _VP, _I, _I,
                                                 ctypes.c_int32, _F, _I, _VP, _VP, _VP, _SZ, _VP, _VP, _VP]
        L.fastar_tempcache_merge_search.argtypes = [ctypes.POINTER(CacheStruct), _VP, _VP, _VP, _I, _I,
                                                    ctypes.c_int32, _F, _I, _VP, _VP, _SZ, _VP, _VP, _VP]
        L.fastar_annsa_quant_attention.argtypes = [_I, _VP, _I, ctypes.POINTER(CacheStruct), _F, _I, _I, _VP, _VP,
                                                   _VP, _VP, _SZ, _VP, _VP]
        L.fastar_annca_quant_attention.argtypes = [_I, _VP, _VP, _VP, _I, _I, _I, _I, _F, _I, _I, _VP, _VP, _VP,
                                                   _SZ, _VP, _VP]
        for name in EXPORTS[7:]:
            getattr(L, name).restype = _I
        _lib = L
    return _lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, where: str):
    if rc != 0:
        raise FastarError(rc, where)


def fastar_check_bounded_wait(polls, status, stream=None):
    """Run the library's bounded-wait error path once (see the C header):
    afterwards `status` holds FASTAR_ERR_TIMEOUT (17) unless it already held
    an error."""
    _check(lib().fastar_check_bounded_wait(int(polls), _p(status), _stream(stream)),
           "fastar_check_bounded_wait")


def fastar_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().fastar_launch_count())


class LaunchTimer:
    """Per-kernel device durations of the library's launches (diagnostic).

    Usage: t = LaunchTimer(n); t.begin(); <calls on the current stream>;
    t.end() -> [(kernel name, ms), ...] in launch order.
    """

    def __init__(self, capacity: int):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        for e in self.events:          # create the underlying CUDA events now
            e.record()
        self.start = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.events])

    def begin(self):
        self.start.record()
        _check(lib().fastar_timing_begin(ctypes.cast(self._handles, ctypes.c_void_p), len(self.events)),
               "fastar_timing_begin")

    def end(self):
        n = int(lib().fastar_timing_end())
        names = [lib().fastar_timing_name(i).decode() for i in range(n)]
        torch.cuda.synchronize()
        out, prev = [], self.start
        for i in range(n):
            out.append((names[i], prev.elapsed_time(self.events[i])))
            prev = self.events[i]
        return out


def fastar_workspace_size(op: int, H: int, N: int, D: int, T: int, B: int, C: int) -> int:
    return int(lib().fastar_workspace_size(op, H, N, D, T, B, C))


def _ws(op, H, N, D, T, B, C, ws, device):
    need = fastar_workspace_size(op, H, N, D, T, B, C)
    if need == 0:
        return None, 0
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
    return ws, ws.numel() * ws.element_size()


def fastar_hash(x, planes, T, B, codes, perm=None, offsets=None, status=None, stream=None):
    """codes [H][T][N] (and optional CSR perm/offsets) of x [H][N][D]."""
    H, N, D = x.shape
    _check(lib().fastar_hash(_dt(x), _p(x), H, N, D, _p(planes), T, B, _p(codes), _p(perm),
                             _p(offsets), None, 0, _p(status), _stream(stream)), "fastar_hash")


def fastar_bucket_csr(codes, B, perm, offsets, status=None, stream=None):
    """perm / offsets of codes [..., N] (leading dims flattened into groups)."""
    N = codes.shape[-1]
    G = codes.numel() // max(N, 1)
    _check(lib().fastar_bucket_csr(_p(codes), G, N, B, _p(perm), _p(offsets), _p(status),
                                   _stream(stream)), "fastar_bucket_csr")


def fastar_hash_many(jobs, planes, T, B, status=None, stream=None):
    """One pass over up to MAX_HASH_JOBS inputs that share H and D.

    jobs: list of (x [H][N][D], codes [H][T][N], perm or None, offsets or
    None); the result equals one fastar_hash call per job."""
    if not 1 <= len(jobs) <= MAX_HASH_JOBS:
        raise ValueError(f"1 to {MAX_HASH_JOBS} jobs")
    arr = (HashJob * len(jobs))()
    H, _, D = jobs[0][0].shape
    for j, (x, codes, perm, offsets) in enumerate(jobs):
        if x.shape[0] != H or x.shape[2] != D or x.dtype != jobs[0][0].dtype:
            raise ValueError("jobs must share H, D and the dtype")
        arr[j] = HashJob(_p(x), x.shape[1], _p(codes), _p(perm), _p(offsets))
    _check(lib().fastar_hash_many(_dt(jobs[0][0]), len(jobs), arr, H, D, _p(planes), T, B, None, 0,
                                  _p(status), _stream(stream)), "fastar_hash_many")


class Cache:
    """Device buffers of one layer's merged cache (allocated once, torch-owned)."""

    def __init__(self, H, C, D, T, B, dtype=torch.bfloat16, device="cuda"):
        self.H, self.C, self.D, self.T, self.B, self.dtype = H, C, D, T, B, dtype
        dev = torch.device(device)
        self.K = torch.zeros(H, C, D, dtype=dtype, device=dev)
        self.V = torch.zeros(H, C, D, dtype=dtype, device=dev)
        self.m = torch.zeros(H, C, dtype=torch.int32, device=dev)
        self.codes = torch.zeros(H, T, C, dtype=torch.int32, device=dev)
        self.last_frame = torch.full((H, C), -1, dtype=torch.int32, device=dev)
        self.size = torch.zeros(H, dtype=torch.int32, device=dev)
        self.inserted = torch.zeros(H, dtype=torch.int64, device=dev)
        self.evicted = torch.zeros(H, dtype=torch.int64, device=dev)
        self.perm = torch.zeros(H, T, C, dtype=torch.int32, device=dev)
        self.offsets = torch.zeros(H, T, (1 << B) + 1, dtype=torch.int32, device=dev)

    BUFFERS = ("K", "V", "m", "codes", "last_frame", "size", "inserted", "evicted", "perm", "offsets")

    @classmethod
    def view(cls, T, B, **buffers):
        """A cache description over existing tensors (nothing is allocated):
        K, V [H][C][D], m, last_frame [H][C], codes, perm [H][T][C], size [H],
        inserted, evicted [H] and offsets [H][T][2^B+1], all given."""
        c = cls.__new__(cls)
        c.H, c.C, c.D = buffers["K"].shape
        c.T, c.B, c.dtype = T, B, buffers["K"].dtype
        for n in cls.BUFFERS:
            setattr(c, n, buffers[n])
        return c

    def struct(self) -> CacheStruct:
        return CacheStruct(self.H, self.D, self.C, self.T, self.B,
                           BF16 if self.dtype == torch.bfloat16 else F32,
                           *[getattr(self, n).data_ptr() for n in self.BUFFERS])

    def snapshot(self) -> dict:
        return {n: getattr(self, n).clone() for n in self.BUFFERS}

    def restore(self, snap: dict):
        for n in self.BUFFERS:
            getattr(self, n).copy_(snap[n], non_blocking=True)

    def save(self, path: str):
        """Write a checkpoint of the cache (every buffer and its shape
        parameters) to `path` with torch.save; a rollout resumed from it
        continues bit for bit as if it had not stopped."""
        torch.save({"shape": (self.H, self.C, self.D, self.T, self.B, str(self.dtype)),
                    "buffers": {n: getattr(self, n).detach().cpu() for n in self.BUFFERS}}, path)

    def load(self, path: str):
        """Restore a checkpoint written by `save` into this cache's buffers
        (same H, C, D, T, B and dtype, or ValueError)."""
        ck = torch.load(path, map_location="cpu")
        if tuple(ck["shape"]) != (self.H, self.C, self.D, self.T, self.B, str(self.dtype)):
            raise ValueError(f"checkpoint of shape {ck['shape']} does not fit this cache")
        for n in self.BUFFERS:
            getattr(self, n).copy_(ck["buffers"][n])

    def nbytes(self) -> int:
        return sum(getattr(self, n).numel() * getattr(self, n).element_size() for n in self.BUFFERS)


def fastar_tempcache_merge(cache: Cache, k_new, v_new, codes_new, F, n_f, first_frame, tau,
                           match_out=None, ws=None, status=None, stream=None, codes_ready=None,
                           rep="last", planes=None, search="prev"):
    """Merge the F frames of a chunk (k_new/v_new [H][F*n_f][D]) into `cache`.

    codes_ready: a torch.cuda.Event after which codes_new and v_new are
    final (fastar_tempcache_merge_ev); None: they are ready on `stream`.
    rep: "last" (the method's representative) or "mean" (the mean-key
    ablation, fastar_tempcache_merge_rep; needs the hash `planes`).
    search: "prev" (the previous frame's groups, the method), "lsh" (every
    earlier group sharing a bucket) or "quant<bits>" (the previous frame's
    groups ranked by their b-bit quantised keys), fastar_tempcache_merge_search."""
    ws, nbytes = _ws(OP_MERGE, cache.H, n_f, cache.D, cache.T, cache.B, cache.C, ws, k_new.device)
    cs = cache.struct()
    if search != "prev":
        if rep != "last":
            raise ValueError("the search over every earlier frame keeps the last key")
        _check(lib().fastar_tempcache_merge_search(
            ctypes.byref(cs), _p(k_new), _p(v_new), _p(codes_new), F, n_f, first_frame, tau, search_code(search),
            _p(match_out), _p(ws), nbytes, _p(status), _stream(stream),
            None if codes_ready is None else codes_ready.cuda_event), "fastar_tempcache_merge_search")
        return
    if rep != "last":
        _check(lib().fastar_tempcache_merge_rep(
            ctypes.byref(cs), _p(k_new), _p(v_new), _p(codes_new), F, n_f, first_frame, tau, REPS[rep],
            _p(planes), _p(match_out), _p(ws), nbytes, _p(status), _stream(stream),
            None if codes_ready is None else codes_ready.cuda_event), "fastar_tempcache_merge_rep")
        return
    args = (ctypes.byref(cs), _p(k_new), _p(v_new), _p(codes_new), F, n_f, first_frame, tau,
            _p(match_out), _p(ws), nbytes, _p(status), _stream(stream))
    if codes_ready is None:
        _check(lib().fastar_tempcache_merge(*args), "fastar_tempcache_merge")
    else:
        _check(lib().fastar_tempcache_merge_ev(*args, codes_ready.cuda_event),
               "fastar_tempcache_merge_ev")


def fastar_annca_prune(q_codes, p_codes, F, n_f, B, kept_idx, kept_cnt, status=None, stream=None):
    """kept_idx [H][F][P] / kept_cnt [H][F] of the prompt tokens per frame."""
    H, T, _ = q_codes.shape
    P = p_codes.shape[2]
    _check(lib().fastar_annca_prune(_p(q_codes), _p(p_codes), H, F, n_f, P, T, B, _p(kept_idx),
                                    _p(kept_cnt), None, 0, _p(status), _stream(stream)),
           "fastar_annca_prune")


def fastar_annca_attention(q, k_p, v_p, kept_idx, kept_cnt, F, n_f, scale, out, ws=None,
                           status=None, stream=None):
    """out [H][F*n_f][D]: cross-attention of each frame over its kept tokens.

    ws: a uint8 device tensor of at least
    fastar_workspace_size(OP_ANNCA, H, F, D, 0, 0, P) bytes; one is allocated
    for the call when it is None."""
    H, Nq, D = q.shape
    P = k_p.shape[1]
    ws, nbytes = _ws(OP_ANNCA, H, F, D, 0, 0, P, ws, q.device)
    _check(lib().fastar_annca_attention(_dt(q), _p(q), _p(k_p), _p(v_p), _p(kept_idx),
                                        _p(kept_cnt), H, F, n_f, P, D, scale, _p(out), _p(ws), nbytes,
                                        _p(status), _stream(stream)), "fastar_annca_attention")


def fastar_annsa_attention_part(q, q_codes, q_perm, q_offsets, cache: Cache, scale, part_base, part_total, ws,
                                status=None, stream=None):
    """Per-table partials of AnnSA over `cache` into slots part_base.. of ws."""
    H, Nq, D = q.shape
    nbytes = ws.numel() * ws.element_size()
    cs = cache.struct()
    _check(lib().fastar_annsa_attention_part(_dt(q), _p(q), _p(q_codes), _p(q_perm), _p(q_offsets), Nq,
                                             ctypes.byref(cs), scale, part_base, part_total, _p(ws), nbytes,
                                             _p(status), _stream(stream)), "fastar_annsa_attention_part")


def fastar_annsa_combine(part_total, ws, out, lse=None, status=None, stream=None):
    """out [H][Nq][D] (and lse) from the part_total partials in ws."""
    H, Nq, D = out.shape
    _check(lib().fastar_annsa_combine(H, Nq, D, part_total, _p(ws), ws.numel() * ws.element_size(), _p(out),
                                      _p(lse), _p(status), _stream(stream)), "fastar_annsa_combine")


def fastar_annsa_attention(q, q_codes, q_perm, q_offsets, cache: Cache, scale, out, lse=None,
                           ws=None, status=None, stream=None):
    """out [H][Nq][D] (and lse [H][Nq]): bucket-restricted attention over `cache`."""
    H, Nq, D = q.shape
    ws, nbytes = _ws(OP_ANNSA, cache.H, Nq, cache.D, cache.T, cache.B, cache.C, ws, q.device)
    cs = cache.struct()
    _check(lib().fastar_annsa_attention(_dt(q), _p(q), _p(q_codes), _p(q_perm), _p(q_offsets), Nq,
                                        ctypes.byref(cs), scale, _p(out), _p(lse), _p(ws), nbytes,
                                        _p(status), _stream(stream)), "fastar_annsa_attention")


def fastar_annsa_quant_attention(q, cache: Cache, scale, topk, bits, out, lse=None, sel_mask=None, ws=None,
                                 status=None, stream=None):
    """out [H][Nq][D]: each query attends its topk live slots of largest
    approximate score under bits-bit quantised keys (sel_mask optional
    [H][Nq][ceil(C/32)] int32 receives the kept slots as bits)."""
    H, Nq, D = q.shape
    ws, nbytes = _ws(OP_QUANT, cache.H, Nq, cache.D, bits, 0, cache.C, ws, q.device)
    cs = cache.struct()
    _check(lib().fastar_annsa_quant_attention(_dt(q), _p(q), Nq, ctypes.byref(cs), scale, topk, bits, _p(out),
                                              _p(lse), _p(sel_mask), _p(ws), nbytes, _p(status), _stream(stream)),
           "fastar_annsa_quant_attention")


def fastar_annca_quant_attention(q, k_p, v_p, scale, topk, bits, out, sel_mask=None, ws=None, status=None,
                                 stream=None):
    """out [H][Nq][D]: each query attends its topk prompt tokens of largest
    approximate score under bits-bit quantised prompt keys."""
    H, Nq, D = q.shape
    P = k_p.shape[1]
    ws, nbytes = _ws(OP_QUANT, H, Nq, D, bits, 0, P, ws, q.device)
    _check(lib().fastar_annca_quant_attention(_dt(q), _p(q), _p(k_p), _p(v_p), H, Nq, P, D, scale, topk, bits,
                                              _p(out), _p(sel_mask), _p(ws), nbytes, _p(status), _stream(stream)),
           "fastar_annca_quant_attention")
