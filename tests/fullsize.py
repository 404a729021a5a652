"""Full-size GPU-vs-oracle comparison, one oracle process per group of heads.

The full-size workloads (the 200-chunk rollout at capacity 32,768 on all 12
heads; the 14B-like layer's 40 heads) are too large for one process of the
fp64 oracle, but heads are independent, so the comparison is split by head:
each spawned process owns some (layer, head) units.  For its units a process
  * draws the inputs with the seeded host generator (workloads.gen) and hands
    them to the test, which runs the library on the GPU;
  * reads the GPU's outputs of each call from shared memory and compares
    them with the oracle run on the same inputs, cascaded as in
    tests/parity.py: codes bit-exact outside the margin bits, CSRs
    bit-exact, NN decisions bit-exact outside listed ones (the oracle then
    continues from the GPU's decisions), cache K, m, codes, last_frame,
    size and counters bit-exact and V within one bf16 ulp, kept lists
    bit-exact, attention within max 1e-2 / mean 1e-3 on the GPU's own state;
  * then takes the GPU's cache state as the state before the next call, so
    that a listed near-tie cannot cascade.
Only the tests import this module (it imports the oracle).
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

ATT_MAX, ATT_MEAN = 1e-2, 1e-3


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bits of float values that are exactly bf16-representable."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bits_to_f64(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp_bf16(x):
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def spec_of(cfg, rows: int):
    """Shared-memory layout of one (layer, head) unit: GPU outputs of a call."""
    T, Nq, P, C, D, F = cfg.T, cfg.Nq, max(cfg.P, 1), cfg.C, cfg.D, cfg.F
    nb = (1 << cfg.B) + 1
    return {"q_codes": ((T, Nq), np.int32), "k_codes": ((T, Nq), np.int32), "p_codes": ((T, P), np.int32),
            "q_perm": ((T, Nq), np.int32), "q_off": ((T, nb), np.int32), "match": ((Nq,), np.int32),
            "K": ((C, D), np.uint16), "V": ((C, D), np.uint16), "m": ((C,), np.int32),
            "codes": ((T, C), np.int32), "last_frame": ((C,), np.int32), "counts": ((3,), np.int64),
            "perm": ((T, C), np.int32), "offsets": ((T, nb), np.int32),
            "kept_idx": ((F, P), np.int32), "kept_cnt": ((F,), np.int32),
            "rows": ((rows,), np.int64), "o_ca": ((rows, D), np.float32), "o_sa": ((rows, D), np.float32),
            "lse": ((rows,), np.float32)}


class ShmArrays:
    """Named numpy arrays in one file mapped by both processes (created or
    attached); a file in a temporary directory rather than /dev/shm, whose
    size some containers cap."""

    def __init__(self, spec, name=None):
        import tempfile
        self.spec = spec
        size, self.off = 0, {}
        for k, (shape, dt) in spec.items():
            self.off[k] = size
            size += (int(np.prod(shape)) * np.dtype(dt).itemsize + 63) // 64 * 64
        self.owner = name is None
        if self.owner:
            where = None
            try:
                sv = os.statvfs("/dev/shm")
                if sv.f_bavail * sv.f_frsize > 8 * size + (1 << 30):
                    where = "/dev/shm"
            except OSError:
                pass
            fd, name = tempfile.mkstemp(prefix="fastar_parity_", suffix=".bin", dir=where)
            os.ftruncate(fd, max(size, 64))
            os.close(fd)
        self.path = name
        self.mm = np.memmap(name, dtype=np.uint8, mode="r+", shape=(max(size, 64),))
        self.a = {k: np.ndarray(shape, dtype=dt, buffer=self.mm, offset=self.off[k])
                  for k, (shape, dt) in spec.items()}

    @property
    def name(self):
        return self.path

    def close(self):
        self.a = {}
        del self.mm
        if self.owner and os.path.exists(self.path):
            os.unlink(self.path)


class Unit:
    """One (layer, head): its input stream, prompt, hyperplanes and the
    oracle state before the next call."""

    def __init__(self, cfg, layer, head, rows_spec, shm_name):
        import oracle as O
        from workloads import HeadStream, planes, prompt
        self.O = O
        self.cfg = cfg.replace(H=1)
        self.layer, self.head = layer, head
        self.stream = HeadStream(self.cfg, layer, head)
        self.planes = planes(self.cfg, layer)
        pk, pv, _ = prompt(self.cfg, layer, head, self.stream.centroids)
        self.pk, self.pv = pk[None], pv[None]
        self.state = O.CacheState.empty(1, cfg.C, cfg.D, cfg.T, cfg.dtype)
        self.shm = ShmArrays(rows_spec, shm_name)
        self.last = None   # inputs of the last frames drawn: k, v, q [1][n][D]
        self.p_checked = False

    def frames(self, n):
        fr = [self.stream.frame() for _ in range(n)]
        k = np.concatenate([f[0] for f in fr])[None]
        v = np.concatenate([f[1] for f in fr])[None]
        q = np.concatenate([f[2] for f in fr])[None]
        self.last = (k, v, q)
        return bf16_bits(k), bf16_bits(v), bf16_bits(q)

    def prompt_bits(self):
        return bf16_bits(self.pk), bf16_bits(self.pv)

    # -- comparisons -------------------------------------------------------
    def _codes(self, gpu, x, rep, what):
        g = np.asarray(gpu, dtype=np.int64).astype(np.uint32)[None]
        o, margin = self.O.hash_codes(x, self.planes, self.cfg.T, self.cfg.B)
        diff = g ^ o
        bad = (diff & ~margin) != 0
        assert not bad.any(), f"{what}: {int(bad.sum())} codes differ outside the margin"
        rep["listed_hash_bits"] += int(sum(bin(int(v)).count("1") for v in margin[margin != 0]))
        rep["differing_listed_bits"] += int(sum(bin(int(v)).count("1") for v in diff[diff != 0]))
        return g

    def _csr(self, perm, off, codes, n, what):
        for t in range(codes.shape[0]):
            op, oo = self.O.bucket_csr(codes[t], 1 << self.cfg.B, n=n)
            np.testing.assert_array_equal(perm[t, :n], op[:n], err_msg=f"{what} perm t{t}")
            np.testing.assert_array_equal(off[t], oo, err_msg=f"{what} offsets t{t}")

    def _gpu_state(self):
        a = self.shm.a
        O = self.O
        cnt = a["counts"]
        return O.CacheState(self.cfg.dtype, bits_to_f64(a["K"])[None], bits_to_f64(a["V"])[None],
                            a["m"].astype(np.int64)[None], a["codes"].astype(np.uint32)[None],
                            a["last_frame"].astype(np.int64)[None], np.array([cnt[0]], np.int64),
                            np.array([cnt[1]], np.int64), np.array([cnt[2]], np.int64))

    def check(self, first_frame, F, full, att_rows):
        """Compare the GPU outputs of the last call (in shared memory) for
        the frames drawn last; `full`: the whole chunk path (else a merge
        of past frames).  Returns the counts of listed / differing items."""
        O, cfg, a = self.O, self.cfg, self.shm.a
        rep = {"listed_hash_bits": 0, "differing_listed_bits": 0, "listed_nn": 0, "differing_listed_nn": 0,
               "v_ulp_diffs": 0, "att_max": 0.0, "att_mean_max": 0.0, "att_rows": 0}
        k, v, q = self.last
        n = F * cfg.n_f
        kc = self._codes(a["k_codes"][:, :n], k, rep, f"L{self.layer} h{self.head} key codes f{first_frame}")
        st_o, match_o, listed = O.tempcache_merge(self.state, k, v, kc, F, cfg.n_f, first_frame, cfg.tau)
        gm = a["match"][:n].astype(np.int64)[None]
        bad = (gm != match_o) & ~listed
        assert not bad.any(), (f"L{self.layer} h{self.head} f{first_frame}: {int(bad.sum())} NN decisions "
                               f"differ outside the listed ones")
        rep["listed_nn"] += int(listed.sum())
        rep["differing_listed_nn"] += int(((gm != match_o) & listed).sum())
        if ((gm != match_o) & listed).any():
            st_o, _, _ = O.tempcache_merge(self.state, k, v, kc, F, cfg.n_f, first_frame, cfg.tau,
                                           match_override=gm)
        g = self._gpu_state()
        what = f"L{self.layer} h{self.head} merge f{first_frame}"
        for name in ("size", "inserted", "evicted"):
            np.testing.assert_array_equal(getattr(g, name), getattr(st_o, name), err_msg=f"{what} {name}")
        sz = int(g.size[0])
        np.testing.assert_array_equal(g.K[0, :sz], st_o.K[0, :sz], err_msg=f"{what} K")
        np.testing.assert_array_equal(g.m[0, :sz], st_o.m[0, :sz], err_msg=f"{what} m")
        np.testing.assert_array_equal(g.codes[0, :, :sz], st_o.codes[0, :, :sz], err_msg=f"{what} codes")
        np.testing.assert_array_equal(g.last_frame[0, :sz], st_o.last_frame[0, :sz], err_msg=f"{what} last_frame")
        dv = np.abs(g.V[0, :sz] - st_o.V[0, :sz])
        assert (dv <= _ulp_bf16(st_o.V[0, :sz]) * 1.0001).all(), f"{what} V beyond one ulp"
        rep["v_ulp_diffs"] += int((dv > 0).sum())
        assert int(g.m[0].sum() + g.evicted[0]) == int(g.inserted[0]), f"{what} count invariant"
        self._csr(a["perm"], a["offsets"], g.codes[0], sz, f"{what} cache CSR")
        if full:
            qc = self._codes(a["q_codes"], q, rep, f"L{self.layer} h{self.head} query codes")
            self._csr(a["q_perm"], a["q_off"], qc[0], cfg.Nq, f"L{self.layer} h{self.head} query CSR")
            if cfg.P:
                pc = self._codes(a["p_codes"][:, :cfg.P], self.pk, rep, f"L{self.layer} h{self.head} prompt codes")
                idx, cnt = O.annca_prune(qc, pc, cfg.F, cfg.n_f)
                np.testing.assert_array_equal(a["kept_cnt"], cnt[0], err_msg="kept counts")
                np.testing.assert_array_equal(a["kept_idx"][:, :cfg.P], idx[0], err_msg="kept lists")
            if att_rows:
                rows = a["rows"][:att_rows].copy()
                for lo in range(0, rows.size, 1024):
                    r = rows[lo:lo + 1024]
                    o_sa, lse = O.annsa_attention(q, qc, g, cfg.scale, rows=r)
                    errs = [np.abs(a["o_sa"][lo:lo + r.size].astype(np.float64) - o_sa[0])]
                    if cfg.P:
                        o_ca = O.annca_attention(q, self.pk, self.pv, idx, cnt, cfg.F, cfg.n_f, cfg.scale, rows=r)
                        errs.append(np.abs(a["o_ca"][lo:lo + r.size].astype(np.float64) - o_ca[0]))
                    for err in errs:
                        mx, mean = float(err.max()), float(err.mean())
                        assert mx <= ATT_MAX and mean <= ATT_MEAN, \
                            f"L{self.layer} h{self.head} attention: max {mx:.3g} mean {mean:.3g}"
                        rep["att_max"] = max(rep["att_max"], mx)
                        rep["att_mean_max"] = max(rep["att_mean_max"], mean)
                    gl = a["lse"][lo:lo + r.size].astype(np.float64)
                    fin = np.isfinite(lse[0])
                    np.testing.assert_array_equal(np.isfinite(gl), fin)
                    assert np.abs(gl[fin] - lse[0][fin]).max(initial=0) <= 1e-3
                rep["att_rows"] += int(rows.size)
        self.state = g   # the next call starts from the GPU's state
        return rep


def _worker(conn):
    units = {}
    try:
        while True:
            msg = conn.recv()
            cmd = msg[0]
            if cmd == "stop":
                break
            try:
                if cmd == "open":
                    _, key, cfg, layer, head, spec, shm_name = msg
                    units[key] = Unit(cfg, layer, head, spec, shm_name)
                    conn.send(("ok", None))
                elif cmd == "frames":
                    _, key, n = msg
                    conn.send(("ok", units[key].frames(n)))
                elif cmd == "prompt":
                    conn.send(("ok", units[msg[1]].prompt_bits()))
                elif cmd == "check":
                    _, key, first, F, full, att_rows = msg
                    conn.send(("ok", units[key].check(first, F, full, att_rows)))
                elif cmd == "close":
                    u = units.pop(msg[1])
                    u.shm.close()
                    conn.send(("ok", None))
            except Exception as e:  # noqa: BLE001 -- reported to the test
                import traceback
                conn.send(("error", f"{e!r}\n{traceback.format_exc()}"))
    finally:
        for u in units.values():
            u.shm.close()
        conn.close()


class Team:
    """Spawned oracle processes (one BLAS thread each) owning (layer, head) units."""

    def __init__(self, workers=None):
        workers = workers or max(1, min(len(os.sched_getaffinity(0)), 16))
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        self.conns, self.procs = [], []
        try:
            for _ in range(workers):
                a, b = ctx.Pipe()
                p = ctx.Process(target=_worker, args=(b,), daemon=True)
                p.start()
                self.conns.append(a)
                self.procs.append(p)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.where = {}
        self.shm = {}

    def open(self, key, cfg, layer, head, rows):
        spec = spec_of(cfg, rows)
        shm = ShmArrays(spec)
        self.shm[key] = shm
        w = len(self.where) % len(self.conns)
        self.where[key] = w
        self.conns[w].send(("open", key, cfg, layer, head, spec, shm.name))

    def call(self, msgs):
        """Send (key, message) pairs, each to the process owning key; return
        the replies in order.  Messages to one process run in order."""
        for key, msg in msgs:
            self.conns[self.where[key]].send(msg)
        out = []
        for key, _ in msgs:
            kind, val = self.conns[self.where[key]].recv()
            if kind != "ok":
                raise AssertionError(f"unit {key}: {val}")
            out.append(val)
        return out

    def wait_open(self, keys):
        for key in keys:
            kind, val = self.conns[self.where[key]].recv()
            if kind != "ok":
                raise AssertionError(f"unit {key}: {val}")

    def close(self):
        for c in self.conns:
            try:
                c.send(("stop",))
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=30)
        for s in self.shm.values():
            s.close()
        self.shm = {}


def sum_reports(reps):
    out = {}
    for r in reps:
        for k, v in r.items():
            out[k] = max(out.get(k, 0), v) if k.startswith("att_max") or k == "att_mean_max" else out.get(k, 0) + v
    return out
