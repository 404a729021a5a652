#!/usr/bin/env python
"""Per-chunk FAST-AR attention path on one GB300: latency, TFLOP/s, roofline.

A step is one pass of the whole per-chunk path over one chunk of the
configured workload.  Default: the 14B-like 720p chunk -- 40 independent
attention layers, each with 40 heads x D 128, 3 latent frames of 3600 tokens
(10,800 queries), a cache of 21 merged past frames (capacity 32,768 groups
per head), 512 prompt tokens, 2 LSH tables x 10 bits.  Per layer:
    hash(queries, new keys, prompt keys) -> TempCache merge (3 frames)
    -> AnnCA prune -> AnnCA attention -> AnnSA attention,
and the 40 layers run one after the other inside the timed region
(ChunkStack.step: each layer's ChunkPath.step, whose cross-attention branch
runs on a second stream beside the merge).  CUDA events on the calling
stream bracket the step.  The merge mutates the caches, so the pre-chunk
snapshot of every layer's cache is restored before every step and L2 is
flushed (a 256 MiB write), both outside the timed window; the inputs of a
step (about 14 GB) are far larger than L2 anyway.  Per-stage and per-kernel
times come from separate passes that run the stages one after the other.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config I] [--shard heads|layers]

Prints one JSON line.  `--impl reference` times the fp64 oracle on the host
cores instead (see oracle_baseline).  Under torchrun each rank runs its
share of the chunk (by default heads [r H / N, (r+1) H / N) of every layer,
no collective on the data path) and the job's time is the slowest rank's.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import CONFIGS, layer_data  # noqa: E402

METRIC = "per-chunk FAST-AR attention ms, effective TFLOP/s, % of GB300 roofline"
# the whole chunk is fixed and split over the ranks, so scaling is strong
SCALING = {"heads": "strong", "layers": "strong"}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=None,
                    help="workload index (default: the 40-layer 14B-like chunk; --recall and --denoise "
                         "default to the one-layer Wan-1.3B-like chunk)")
    ap.add_argument("--shard", default="heads", choices=["heads", "layers"],
                    help="multi-GPU split of the chunk: heads of every layer (default) or whole layers")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only this many of the workload's layers (a small case for profilers; the "
                         "printed line then describes that many layers)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-rollout", action="store_true",
                    help="skip the 200-chunk rollout measurement appended to the default line")
    ap.add_argument("--rep", default="last", choices=["last", "mean"],
                    help="TempCache representative: last key (the method) or mean key (ablation)")
    ap.add_argument("--search", default="prev",
                    help="TempCache search: prev (the previous frame's groups, the method), lsh (every earlier "
                         "group sharing an LSH bucket) or quant<bits> (the previous frame's groups ranked by "
                         "their quantised keys)")
    ap.add_argument("--quant", type=str, default="",
                    help="comma-separated bits (e.g. 2,4,8,16): the quantised matcher (TempCache-Quant, "
                         "AnnCA-Quant, AnnSA-Quant) per chunk, recall and density (one JSON line)")
    ap.add_argument("--denoise", type=int, default=0,
                    help="time the S denoising steps of one chunk (dense for the first 30%%) against "
                         "all-dense and all-sparse schedules (one JSON line)")
    ap.add_argument("--recall", action="store_true",
                    help="sweep tau, T and B: recall and density of AnnSA and AnnCA (one JSON line)")
    return ap.parse_args(argv)


def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def shard(cfg, rank: int, world: int, mode: str = "heads"):
    """The (layers, heads) of the chunk that rank `rank` of `world` runs.

    heads:  every layer, heads [r H / N, (r+1) H / N) (each GPU owns its
            heads' cache slices; heads share nothing on the path);
    layers: layers r, r + N, r + 2N, ... with every head.
    Over all ranks every (layer, head) of the chunk is run exactly once."""
    if mode == "heads":
        if world > cfg.H:
            raise ValueError(f"{world} ranks for {cfg.H} heads")
        return list(range(cfg.layers)), list(range(rank * cfg.H // world, (rank + 1) * cfg.H // world))
    if mode == "layers":
        if world > cfg.layers:
            raise ValueError(f"{world} ranks for {cfg.layers} layers")
        return list(range(rank, cfg.layers, world)), list(range(cfg.H))
    raise ValueError(mode)


def config_dict(cfg, args, world):
    """The workload description printed by both arms (identical keys)."""
    return {"workload": cfg.name, "layers": cfg.layers, "H": cfg.H, "D": cfg.D, "n_f": cfg.n_f, "F": cfg.F,
            "Nq": cfg.Nq, "P": cfg.P, "T": cfg.T, "B": cfg.B, "C": cfg.C, "tau": cfg.tau,
            "past_frames": cfg.past_frames, "representative": args.rep, "search": args.search,
            "l2": "flushed before every step (256 MiB write); inputs larger than L2",
            "parallelism": (f"{args.shard}-sharded x{world}, no collective on the data path" if world > 1
                            else "single GPU")}


def job_max(x: float, world: int, device) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- clocks
class Clocks:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc, self.path, self.gpu = None, None, gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # wait for the first sample so that the sampler runs before timing starts
        for _ in range(100):
            time.sleep(0.05)
            if os.path.getsize(self.path) > 0:
                break

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    def stop(self):
        """Median SM clock and active throttle reasons of the samples taken in window()."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        import datetime as _dt
        sm_in, sm_all, smax, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    sm = float(parts[2])
                    smax = float(parts[3])
                except ValueError:
                    continue
                inside = t0 is None or (t0 - 0.05 <= ts <= t1 + 0.05)
                sm_all.append(sm)
                if not inside:
                    continue
                sm_in.append(sm)
                for n, v in zip(names, parts[6:10]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        use = sm_in if sm_in else sm_all
        return {"sm_mhz": statistics.median(use) if use else None, "sm_max_mhz": smax,
                "samples": len(sm_in), "samples_run": len(sm_all), "reasons": sorted(reasons)}


# ----------------------------------------------------------------- oracle leg
# The oracle (numpy fp64) is timed on the host cores, one process per core
# (spawned, each with one BLAS thread), each process owning one (layer, head)
# unit of the chunk: it draws that head's frames with the seeded generator,
# merges the past frames (set-up, untimed), then times the whole per-chunk
# path of its unit -- hash of queries, new keys and prompt keys, query CSR,
# TempCache merge of the chunk's frames, cache CSR, AnnCA prune, AnnCA,
# AnnSA -- once per step from the same pre-chunk state.  A step is one unit
# on every process at once; the chunk's time is extrapolated from the
# throughput (units per second) to all its (layer, head) units.

def _oracle_unit_setup(cfg, layer: int, head: int):
    import oracle as O
    cfg = cfg.replace(H=1)
    d = layer_data(cfg, layer=layer, chunks=1, heads=[head])
    st = O.CacheState.empty(1, cfg.C, cfg.D, cfg.T, cfg.dtype)
    f = 0
    while f < cfg.past_frames:
        nF = min(cfg.F, cfg.past_frames - f)
        k = np.concatenate(d.past_k[f:f + nF], axis=1)
        v = np.concatenate(d.past_v[f:f + nF], axis=1)
        kc, _ = O.hash_codes(k, d.planes, cfg.T, cfg.B)
        st, _, _ = O.tempcache_merge(st, k, v, kc, nF, cfg.n_f, f, cfg.tau)
        f += nF
    return cfg, d, st


def _oracle_unit_chunk(cfg, d, st) -> float:
    """The oracle's whole per-chunk path for one (layer, head); seconds."""
    import oracle as O
    q, k, v = d.chunk_q[0], d.chunk_k[0], d.chunk_v[0]
    t0 = time.perf_counter()
    qc, _ = O.hash_codes(q, d.planes, cfg.T, cfg.B)
    O.bucket_csr(qc, 1 << cfg.B)
    kc, _ = O.hash_codes(k, d.planes, cfg.T, cfg.B)
    pc, _ = O.hash_codes(d.prompt_k, d.planes, cfg.T, cfg.B)
    st2, _, _ = O.tempcache_merge(st, k, v, kc, cfg.F, cfg.n_f, cfg.past_frames, cfg.tau)
    O.bucket_csr(st2.codes, 1 << cfg.B)
    idx, cnt = O.annca_prune(qc, pc, cfg.F, cfg.n_f)
    O.annca_attention(q, d.prompt_k, d.prompt_v, idx, cnt, cfg.F, cfg.n_f, cfg.scale)
    O.annsa_attention(q, qc, st2, cfg.scale)
    return time.perf_counter() - t0


def _oracle_worker(conn, cfg, layer, head):
    """Process body: set up one unit, then time it once per 'go'."""
    try:
        cfg, d, st = _oracle_unit_setup(cfg, layer, head)
        conn.send(("ready", None))
        while True:
            msg = conn.recv()
            if msg != "go":
                break
            conn.send(("done", _oracle_unit_chunk(cfg, d, st)))
    except Exception as e:  # reported to the parent, which raises
        conn.send(("error", repr(e)))
    finally:
        conn.close()


class OracleTeam:
    """One spawned process per host core, each owning a (layer, head) unit."""

    def __init__(self, cfg, workers: int):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        self.units = [(w // cfg.H % cfg.layers, w % cfg.H) for w in range(workers)]
        self.conns, self.procs = [], []
        try:
            for layer, head in self.units:
                a, b = ctx.Pipe()
                p = ctx.Process(target=_oracle_worker, args=(b, cfg, layer, head), daemon=True)
                p.start()
                self.conns.append(a)
                self.procs.append(p)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        t0 = time.perf_counter()
        self._collect("ready")
        self.setup_s = time.perf_counter() - t0

    def _collect(self, want):
        out = []
        for c in self.conns:
            kind, val = c.recv()
            if kind != want:
                raise RuntimeError(f"oracle worker: {kind} {val}")
            out.append(val)
        return out

    def step(self):
        """One unit on every process at once: (wall seconds, per-unit seconds)."""
        t0 = time.perf_counter()
        for c in self.conns:
            c.send("go")
        per = self._collect("done")
        return time.perf_counter() - t0, per

    def close(self):
        for c in self.conns:
            try:
                c.send("stop")
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=10)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo; "unknown" elsewhere)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                return v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                k, _, v = line.partition(":")
                if k.strip().lower() in ("model name", "cpu model", "hardware") and v.strip():
                    return v.strip()
            fh.seek(0)
            for line in fh:
                k, _, v = line.partition(":")
                if k.strip().lower() == "cpu part":
                    return "cpu part " + v.strip()
    except OSError:
        pass
    return "unknown"


def oracle_baseline(cfg, timed_steps: int, warm_steps: int):
    """Time the oracle on the host cores (see above).  Returns the JSON
    object of the measurement: per-chunk ms extrapolated from the measured
    unit throughput, the measured step times and what the sample was."""
    workers = min(host_cores(), cfg.layers * cfg.H)
    team = OracleTeam(cfg, workers)
    try:
        for _ in range(warm_steps):
            team.step()
        walls, units = [], []
        for _ in range(timed_steps):
            w, per = team.step()
            walls.append(w)
            units.extend(per)
    finally:
        team.close()
    step_s = statistics.mean(walls)
    units_per_chunk = cfg.layers * cfg.H
    chunk_ms = step_s * units_per_chunk / workers * 1e3
    return {"value": chunk_ms, "unit": "ms/chunk", "cores": workers, "kind": "oracle",
            "ms_per_step": step_s * 1e3, "steps": timed_steps, "warmup": warm_steps,
            "unit_ms_mean": statistics.mean(units) * 1e3, "setup_s": team.setup_s,
            # the chunk on one core: every process is one thread (one BLAS
            # thread), so a unit's time is its one-core time
            "one_core_ms_per_chunk": statistics.mean(units) * 1e3 * units_per_chunk,
            "cpu_model": host_cpu_model(), "host_cores": host_cores(),
            "sample": (f"{workers} (layer, head) units of the {cfg.layers}-layer x {cfg.H}-head chunk, one per "
                       f"process (one BLAS thread each, {workers} processes on {host_cores()} host cores); a step "
                       f"times every process's unit once (hash, query CSR, merge of the chunk's {cfg.F} frames, "
                       f"cache CSR, prune, AnnCA, AnnSA; past frames merged untimed); per chunk = step time x "
                       f"{units_per_chunk} units / {workers}")}


def run_reference(args, cfg):
    rank, world, _ = rank_info()
    if rank != 0:
        return
    timed, warm = min(args.steps, 8), min(args.warmup, 1)
    t_run = time.perf_counter()
    ob = oracle_baseline(cfg, timed, warm)
    t_run = time.perf_counter() - t_run
    line = {"impl": "reference", "metric": METRIC, "value": ob["value"], "unit": "ms/chunk",
            "n_gpus": args.gpus, "steps": timed, "warmup": warm,
            "ms_per_step": ob["ms_per_step"], "higher_is_better": False, "scaling": SCALING[args.shard],
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg, args, world),
            "extrapolated_to_chunk": {"value": ob["value"], "unit": "ms/chunk",
                                      "from": "unit throughput of the timed steps (see cpu_baseline.sample)"},
            "cpu_baseline": {k: ob[k] for k in ("value", "unit", "cores", "kind", "sample", "unit_ms_mean", "one_core_ms_per_chunk",
                                                "cpu_model", "host_cores", "setup_s")},
            "wall_s": t_run,
            "e2e": {"value": ob["value"], "unit": "ms/chunk", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU leg
def _pairs_union(q_codes, c_codes, sizes, B):
    """Allowed (query, slot) pairs of one layer, by inclusion-exclusion over
    the tables: a pair is allowed iff its codes agree in some table, so
    |union| = sum over non-empty table subsets S of (-1)^(|S|+1) times the
    number of pairs whose codes agree in every table of S, counted from
    joint code histograms.  q_codes [H][T][Nq], c_codes [H][T][C] (int32,
    device), sizes [H] live slots.  Returns (total, per-table pairs not
    already allowed by an earlier table)."""
    import itertools

    import torch
    H, T, Nq = q_codes.shape
    C = c_codes.shape[2]
    live = torch.arange(C, device=c_codes.device)[None, :] < sizes[:, None].long()
    hq = torch.arange(H, device=q_codes.device)[:, None].expand(H, Nq)
    hc = torch.arange(H, device=c_codes.device)[:, None].expand(H, C)

    def agree(S):
        kq, kc = hq.long(), hc.long()
        for t in S:
            kq = (kq << B) | q_codes[:, t].long()
            kc = (kc << B) | c_codes[:, t].long()
        kc = kc[live]
        uq, cq = torch.unique(kq.reshape(-1), return_counts=True)
        uc, cc = torch.unique(kc, return_counts=True)
        idx = torch.searchsorted(uc, uq).clamp_max(max(uc.numel() - 1, 0))
        hit = uc[idx] == uq if uc.numel() else torch.zeros_like(uq, dtype=torch.bool)
        return int((cq[hit] * cc[idx[hit]]).sum())

    cache = {}

    def count(S):
        if S not in cache:
            cache[S] = agree(S)
        return cache[S]

    def union(tables):
        tot = 0
        for r in range(1, len(tables) + 1):
            for S in itertools.combinations(tables, r):
                tot += (-1) ** (r + 1) * count(S)
        return tot

    by_table = [union(tuple(range(t + 1))) - union(tuple(range(t))) if t else count((0,)) for t in range(T)]
    return sum(by_table), by_table


def annsa_tiles(path, n_live):
    """Key tiles the AnnSA kernel walks for this layer (its work performed):
    per table t, the queries in table-t bucket order are cut into tiles of
    128; a tile walks the cache slots of every table-t bucket from its first
    query's to its last query's, 64 at a time.  Returns the number of
    (128-query x 64-key) tiles."""
    import torch
    H, T, Nq = path.q_codes.shape
    nb = 1 << path.B
    tiles = 0
    idx = torch.arange(0, Nq, 128, device=path.q_codes.device)
    last = torch.clamp(idx + 127, max=Nq - 1)
    for t in range(T):
        perm = path.q_perm[:, t].long()
        codes = path.q_codes[:, t].long()
        c_lo = torch.gather(codes, 1, perm[:, idx])
        c_hi = torch.gather(codes, 1, perm[:, last])
        off = path.cache.offsets[:, t].long()
        kb = torch.gather(off, 1, c_lo).clamp(max=n_live[:, None])
        ke = torch.gather(off, 1, (c_hi + 1).clamp(max=nb)).clamp(max=n_live[:, None])
        tiles += int(((ke - kb).clamp(min=0) + 63).div(64, rounding_mode="floor").sum())
    return tiles


def layer_work(cfg, path, snap):
    """Algorithmic work of one layer's chunk (from its outputs after a step).

    Bytes count each input read once and each output written once
    (element size e); flops are 2 M N K for a GEMM and 4 D per allowed
    (query, key) pair of attention.  Returns a dict of stage bytes / flops,
    per-kernel models (bytes and flops of all launches of the layer) and
    counts."""
    import torch
    H, D, T, Nq, P, n_f, F = path.H, cfg.D, cfg.T, cfg.Nq, cfg.P, cfg.n_f, cfg.F
    e = 2 if cfg.dtype == "bf16" else 4
    size = path.cache.size.long()
    n_live = int(size.sum())
    kept = int(path.kept_cnt.long().sum())
    kept_tiles = int(((path.kept_cnt.long() + 63) // 64).sum())
    rows = H * (2 * Nq + P)
    C = path.C
    lf0 = snap["last_frame"]
    ar = torch.arange(C, device=lf0.device)[None]
    cand = [int(((lf0 == cfg.past_frames - 1) & (ar < snap["size"][:, None])).sum())]
    mt = path.match.view(H, F, n_f).long()
    hh = torch.arange(H, device=mt.device)[:, None].expand(H, n_f)
    merge_b, apply_b, nn_fl, nn_b = 0, 0, 0, 0
    for fi in range(F):
        m = mt[:, fi]
        matched = m >= 0
        n_matched = int(matched.sum())
        groups = int(torch.unique((hh * C + m)[matched]).numel())
        new = H * n_f - n_matched
        touched = groups + new
        nn_fl += 2 * D * n_f * cand[-1]
        nn_b += (H * n_f + cand[-1]) * D * e
        # apply: new k, v read; matched groups' V read; K, V, m, last_frame
        # and codes of every touched slot written
        apply_b += 2 * H * n_f * D * e + groups * D * e + touched * (2 * D * e + 8 + T * 4)
        if fi + 1 < F:
            cand.append(touched)
    csr_b = n_live * T * (4 + 4) + H * T * ((1 << cfg.B) + 1) * 4
    merge_b = nn_b + apply_b + csr_b
    pairs, pairs_t = _pairs_union(path.q_codes, path.cache.codes, size, cfg.B)
    sa_tiles = annsa_tiles(path, size)
    by = {"hash": rows * (D * e + T * 4) + T * cfg.B * D * e,
          "merge": merge_b,
          "prune": H * T * (Nq + P) * 4 + H * F * P * 4,
          "annca": 2 * H * Nq * D * e + kept * 2 * D * e + H * F * P * 4,
          "annsa": (2 * H * Nq * D * e + H * T * Nq * 4 + n_live * (2 * D * e + 4 + T * 4)
                    + H * Nq * 4)}
    fl = {"hash": 2 * rows * T * cfg.B * D, "merge": nn_fl, "prune": 0,
          "annca": 4 * D * n_f * kept, "annsa": 4 * D * pairs}
    kern = {
        "nn_tc": {"flops": nn_fl, "bytes": nn_b},
        "apply": {"flops": 0, "bytes": apply_b},
        "annca_tc": {"flops": fl["annca"], "bytes": by["annca"],
                     "work_flops": 4 * 128 * 64 * D * sum(int(x) for x in
                                                          ((path.kept_cnt.long() + 63) // 64).view(-1).tolist())
                     * ((n_f + 127) // 128)},
        # the stage's algorithmic bytes (Q, live K/V/m/codes, O, lse, q codes
        # each once) and its allowed-pair flops
        "annsa_tc": {"flops": fl["annsa"], "bytes": by["annsa"],
                     "work_flops": 4 * 128 * 64 * D * sa_tiles},
        "annca_compact": {"flops": 0, "bytes": 2 * kept * D * e + 2 * kept_tiles * 64 * D * e + (kept + H * F) * 4},
        "hash_tc": {"flops": fl["hash"], "bytes": rows * (D * e + T * 4)},
    }
    return {"bytes": by, "flops": fl, "kern": kern,
            "stats": {"n_live": n_live, "kept": kept, "allowed_pairs": pairs, "allowed_pairs_by_table": pairs_t,
                      "annsa_key_tiles": sa_tiles, "density_den": Nq * n_live}}


KERNEL_SOURCES = {"nn_tc": "nn_tc.cu", "annca_tc": "attention_tc.cu", "annsa_tc": "attention_tc.cu",
                  "hash_tc": "hash_tc.cu", "apply": "tempcache.cu"}


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic_<kernel>_<workload>.txt), or None when there is none
    or the kernel's source has changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.txt")
    src = KERNEL_SOURCES.get(kernel)
    if not src or not os.path.exists(path):
        return None
    vals = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    with open(os.path.join(ROOT, "merged_attention_autoregressive_gb300", "csrc", src), "rb") as fh:
        sha = hashlib.sha256(fh.read()).hexdigest()[:16]
    if vals.get("source_sha256_16") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def dense_sdpa(q, K, V, kp, vp, reps=5):
    """Dense attention of one layer's chunk: torch SDPA over the unmerged
    history and over the whole prompt (bf16).  Returns ms per layer."""
    import torch
    import torch.nn.functional as Fn

    def run():
        Fn.scaled_dot_product_attention(q[None], K[None], V[None])
        if kp.shape[1]:
            Fn.scaled_dot_product_attention(q[None], kp[None], vp[None])
    for _ in range(2):
        run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        run()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


def dense_ours(q, K, V, kp, vp, n_f, F, reps=5):
    """Dense attention of one layer's chunk through this library's own kernels.

    A cache in which every key of the unmerged history is its own group
    (m = 1) and every code is 0 (one table of one bit, one bucket) makes
    AnnSA dense attention over the history; a kept list holding every
    prompt token makes AnnCA dense cross-attention.  The cache buffers are
    caller-owned, so they are written directly here (set-up, untimed).  This
    measures the attention kernels on dense work: their tensor-core
    throughput against the measured bf16 peak, beside torch SDPA."""
    import torch
    import torch.nn.functional as Fn

    import merged_attention_autoregressive_gb300 as fa
    H, Nq, D = q.shape
    P = kp.shape[1]
    n = K.shape[1]
    c = fa.Cache(H, n, D, 1, 1, q.dtype)
    c.K.copy_(K)
    c.V.copy_(V)
    c.m.fill_(1)
    c.last_frame.zero_()
    c.size.fill_(n)
    c.inserted.fill_(n)
    c.perm[:, 0].copy_(torch.arange(n, dtype=torch.int32, device="cuda"))
    c.offsets[:, 0] = torch.tensor([0, n, n], dtype=torch.int32, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    q_codes = torch.zeros(H, 1, Nq, **i32)
    q_perm = torch.arange(Nq, **i32).repeat(H, 1, 1).contiguous()
    q_off = torch.tensor([0, Nq, Nq], **i32).repeat(H, 1, 1).contiguous()
    kept_idx = torch.arange(max(P, 1), **i32).repeat(H, F, 1).contiguous()
    kept_cnt = torch.full((H, F), P, **i32)
    o_sa = torch.empty(H, Nq, D, dtype=q.dtype, device="cuda")
    o_ca = torch.empty(H, Nq, D, dtype=q.dtype, device="cuda")
    lse = torch.empty(H, Nq, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, **i32)
    ws_sa = torch.empty(max(1, fa.fastar_workspace_size(fa.OP_ANNSA, H, Nq, D, 1, 1, n)), dtype=torch.uint8,
                        device="cuda")
    ws_ca = torch.empty(max(1, fa.fastar_workspace_size(fa.OP_ANNCA, H, F, D, 1, 1, P)), dtype=torch.uint8,
                        device="cuda")
    scale = D ** -0.5
    stream = torch.cuda.current_stream()

    def sa():
        fa.fastar_annsa_attention(q, q_codes, q_perm, q_off, c, scale, o_sa, lse, ws=ws_sa, status=st)

    def ca():
        if P:
            fa.fastar_annca_attention(q, kp, vp, kept_idx, kept_cnt, F, n_f, scale, o_ca, ws=ws_ca, status=st)

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    ms_sa, ms_ca = timed(sa), timed(ca)
    assert int(st.item()) == 0, fa.STATUS.get(int(st.item()))
    # agreement with SDPA on a few heads (bf16 outputs of both)
    err = 0.0
    for h in range(min(H, 2)):
        ref = Fn.scaled_dot_product_attention(q[h][None], K[h][None], V[h][None])[0]
        err = max(err, float((o_sa[h].float() - ref.float()).abs().max()))
        if P:
            ref = Fn.scaled_dot_product_attention(q[h][None], kp[h][None], vp[h][None])[0]
            err = max(err, float((o_ca[h].float() - ref.float()).abs().max()))
    pk = peaks()
    fl_sa, fl_ca = 4 * D * H * Nq * n, 4 * D * H * Nq * P
    out = {"impl": "this library's AnnSA / AnnCA kernels, one bucket (dense)", "keys": n,
           "ms": ms_sa + ms_ca, "ms_self": ms_sa, "ms_cross": ms_ca,
           "tflops_self": fl_sa / ms_sa / 1e9,
           "frac_self": fl_sa / ms_sa / 1e9 / pk["bf16_tflops"],
           "tflops_cross": fl_ca / ms_ca / 1e9 if P else None,
           "frac_cross": fl_ca / ms_ca / 1e9 / pk["bf16_tflops"] if P else None,
           "peak_tflops": pk["bf16_tflops"], "peak_of": "measured bf16 burst",
           "max_abs_err_vs_sdpa": err}
    del c
    torch.cuda.empty_cache()
    return out


class LayerSource:
    """The frames, prompt and hyperplanes of one layer, as device tensors of
    the heads `heads`: drawn on the device (workloads.gen_device) unless the
    workload's prompt has its own clusters (the long-prompt workload, whose
    relevance labels come from the host generator)."""

    def __init__(self, cfg, layer, heads, device="cuda"):
        import torch
        self.cfg, self.hs, self.dev = cfg, slice(heads[0], heads[-1] + 1), device
        self.tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        self.rel = None
        if cfg.prompt_clusters:
            self.np = layer_data(cfg, layer=layer, chunks=1)
            self.next = 0
            self.rel = self.np.prompt_rel[self.hs]
        else:
            from workloads.gen_device import DeviceLayerStream
            self.np = None
            self.ds = DeviceLayerStream(cfg, layer, device)

    def _dev(self, a):
        import torch
        return torch.from_numpy(np.ascontiguousarray(a[self.hs])).to(self.dev, self.tdt)

    def planes(self):
        import torch
        if self.np is not None:
            return torch.from_numpy(self.np.planes).to(self.dev, self.tdt)
        return self.ds.planes()

    def frames(self, n):
        """(k, v, q) of the next n frames, concatenated over frames: [H][n n_f][D]."""
        import torch
        if self.np is not None:
            cfg = self.cfg
            f0 = self.next
            self.next += n
            if f0 >= cfg.past_frames:
                c = (f0 - cfg.past_frames) // cfg.F
                return self._dev(self.np.chunk_k[c]), self._dev(self.np.chunk_v[c]), self._dev(self.np.chunk_q[c])
            cat = lambda xs: self._dev(np.concatenate(xs, axis=1))  # noqa: E731
            return cat(self.np.past_k[f0:f0 + n]), cat(self.np.past_v[f0:f0 + n]), None
        fr = [self.ds.frame() for _ in range(n)]
        return tuple(torch.cat([f[i][self.hs] for f in fr], dim=1).contiguous() for i in range(3))

    def prompt(self):
        if self.np is not None:
            return self._dev(self.np.prompt_k), self._dev(self.np.prompt_v)
        kp, vp = self.ds.prompt()
        return kp[self.hs].contiguous(), vp[self.hs].contiguous()


def prepare_stack(cfg, args, layers, heads, keep_history=False):
    """Caches of the rank's layers with their past frames merged, and the
    chunk inputs.  Returns (stack, inputs, sources, history of the first
    layer (K, V of every unmerged key) or None)."""
    import torch

    from merged_attention_autoregressive_gb300.path import ChunkStack
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    stack = ChunkStack(len(layers), len(heads), cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau, tdt,
                       rep=args.rep, search=args.search)
    inputs, sources, hist = [], [], None
    for i, layer in enumerate(layers):
        src = LayerSource(cfg, layer, heads)
        path = stack.paths[i]
        path.planes.copy_(src.planes())
        hk, hv = [], []
        f = 0
        while f < cfg.past_frames:
            nF = min(cfg.F, cfg.past_frames - f)
            k, v, _ = src.frames(nF)
            path.merge(k, v, f, F=nF)
            if keep_history and i == 0:
                hk.append(k)
                hv.append(v)
            f += nF
        k, v, q = src.frames(cfg.F)
        kp, vp = src.prompt()
        inputs.append((q, k, v, kp, vp))
        sources.append(src)
        if keep_history and i == 0:
            hist = (torch.cat(hk + [k], dim=1), torch.cat(hv + [v], dim=1))
        torch.cuda.synchronize()
        assert int(path.status.item()) == 0, f"layer {layer}: device status {int(path.status.item())}"
    return stack, inputs, sources, hist


def run_stages(path, x, first, cfg, args, ev):
    """The five stages of one layer one after the other on the current
    stream, recording ev[0..5] around them (per-stage times)."""
    import torch

    import merged_attention_autoregressive_gb300 as fa
    q, k, v, kp, vp = x
    stream = torch.cuda.current_stream()
    st = path.status
    ev[0].record(stream)
    jobs = [(q, path.q_codes, path.q_perm, path.q_offsets), (k, path.k_codes, None, None)]
    if cfg.P:
        jobs.append((kp, path.p_codes, None, None))
    fa.fastar_hash_many(jobs, path.planes, cfg.T, cfg.B, status=st)
    ev[1].record(stream)
    fa.fastar_tempcache_merge(path.cache, k, v, path.k_codes, cfg.F, cfg.n_f, first, cfg.tau,
                              match_out=path.match, ws=path.ws_merge, status=st, rep=args.rep, planes=path.planes,
                              search=args.search)
    ev[2].record(stream)
    fa.fastar_annca_prune(path.q_codes, path.p_codes[:, :, :cfg.P], cfg.F, cfg.n_f, cfg.B, path.kept_idx,
                          path.kept_cnt, status=st)
    ev[3].record(stream)
    fa.fastar_annca_attention(q, kp, vp, path.kept_idx, path.kept_cnt, cfg.F, cfg.n_f, path.scale, path.o_ca,
                              ws=path.ws_annca, status=st)
    ev[4].record(stream)
    fa.fastar_annsa_attention(q, path.q_codes, path.q_perm, path.q_offsets, path.cache, path.scale, path.o_sa,
                              path.lse, ws=path.ws_annsa, status=st)
    ev[5].record(stream)


def run_ours(args, cfg):
    import torch
    import torch.distributed as dist

    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build as fbuild

    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fbuild.build()
    fa.lib()
    layers, heads = shard(cfg, rank, world, args.shard)
    want_dense = not args.no_dense and rank == 0 and cfg.dtype == "bf16"
    t_prep = time.perf_counter()
    stack, inputs, sources, hist = prepare_stack(cfg, args, layers, heads, keep_history=want_dense)
    snaps = [p.cache.snapshot() for p in stack.paths]
    t_prep = time.perf_counter() - t_prep
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    first = cfg.past_frames
    stages = ["hash", "merge", "prune", "annca", "annsa"]

    def prep():
        for p, sn in zip(stack.paths, snaps):
            p.cache.restore(sn)
        flush.fill_(1)

    def check():
        for p in stack.paths:
            assert int(p.status.item()) == 0, fa.STATUS.get(int(p.status.item()))

    for _ in range(max(3, args.warmup)):
        prep()
        stack.step(inputs, first)
    torch.cuda.synchronize()
    check()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = Clocks(local)
    n0 = fa.fastar_launch_count()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0 = time.time()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        prep()
        evs[i][0].record(stream)
        stack.step(inputs, first)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks.window(t0, time.time())
    clk = clocks.stop()
    launches = fa.fastar_launch_count() - n0
    check()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms = statistics.mean(step_ms)
    # the job's time per chunk is its slowest rank's; the ranks together ran
    # every (layer, head) of the chunk once per step
    value = job_max(ms, world, "cuda")
    ms_median = job_max(statistics.median(step_ms), world, "cuda")

    # the same steps with L2 left warm (the caches are restored, nothing is
    # flushed), beside the flushed measurement above
    warm_ms = []
    for _ in range(min(args.steps, 5)):
        for p, sn in zip(stack.paths, snaps):
            p.cache.restore(sn)
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        stack.step(inputs, first)
        w1.record(stream)
        torch.cuda.synchronize()
        warm_ms.append(w0.elapsed_time(w1))
    check()
    l2_warm = job_max(statistics.mean(warm_ms), world, "cuda")

    # per-stage times: the stages of every layer one after the other
    n_ss = min(args.steps, 3)
    stage_ms = {s_: 0.0 for s_ in stages}
    for _ in range(n_ss):
        prep()
        sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in stack.paths]
        for p, x, ev in zip(stack.paths, inputs, sevs):
            run_stages(p, x, first, cfg, args, ev)
        torch.cuda.synchronize()
        for j, s_ in enumerate(stages):
            stage_ms[s_] += sum(ev[j].elapsed_time(ev[j + 1]) for ev in sevs) / n_ss
    check()

    # per-kernel durations: the library's launch timer (events on the launch
    # stream after every kernel) over the same sequential stages
    timer = fa.LaunchTimer(48 * len(stack.paths) + 16)
    per_kernel = {}
    n_ts = min(args.steps, 2)
    for _ in range(n_ts):
        prep()
        sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in stack.paths]
        timer.begin()
        for p, x, ev in zip(stack.paths, inputs, sevs):
            run_stages(p, x, first, cfg, args, ev)
        for name, ms_k in timer.end():
            per_kernel.setdefault(name, []).append(ms_k)
    kernels = {k: {"launches_per_step": len(v) / n_ts, "avg_ms": statistics.mean(v),
                   "ms_per_step": sum(v) / n_ts} for k, v in per_kernel.items()}
    check()

    # end to end through the public call with host buffers (pinned): every
    # layer's inputs copied in and both outputs copied out inside the window
    def pinned_copy(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h
    hin = [tuple(pinned_copy(t) for t in x) for x in inputs]
    hout = [(torch.empty(p.o_ca.shape, dtype=p.o_ca.dtype, pin_memory=True),
             torch.empty(p.o_sa.shape, dtype=p.o_sa.dtype, pin_memory=True)) for p in stack.paths]
    h2d = sum(t.numel() * t.element_size() for x in hin for t in x)
    d2h = sum(t.numel() * t.element_size() for x in hout for t in x)
    e2e = []
    for i in range(args.steps + 2):
        prep()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        stack.step_host(hin, hout, first, dev_in=inputs)
        s1.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            e2e.append(s0.elapsed_time(s1))
    check()
    e2e_ms = job_max(statistics.mean(e2e), world, "cuda")
    # the window is bound by the host copies (13.7 GB in, 8.8 GB out per
    # chunk of the 14B-like workload); on a box whose host link other jobs
    # share, single chunks stall on it, so the median and the fastest chunk
    # are given beside the mean
    e2e_med = job_max(statistics.median(e2e), world, "cuda")
    e2e_min = job_max(min(e2e), world, "cuda")
    del hin, hout

    # algorithmic work of the step (from the last step's outputs), summed
    # over this rank's layers
    by = {s_: 0 for s_ in stages}
    fl = {s_: 0 for s_ in stages}
    kern, stats = {}, {}
    for p, sn in zip(stack.paths, snaps):
        w = layer_work(cfg, p, sn)
        for s_ in stages:
            by[s_] += w["bytes"][s_]
            fl[s_] += w["flops"][s_]
        for k_, m_ in w["kern"].items():
            d_ = kern.setdefault(k_, {})
            for kk, vv in m_.items():
                d_[kk] = d_.get(kk, 0) + vv
        for k_, v_ in w["stats"].items():
            if isinstance(v_, list):
                stats[k_] = [a + b for a, b in zip(stats.get(k_, [0] * len(v_)), v_)]
            else:
                stats[k_] = stats.get(k_, 0) + v_
    stats["density"] = stats.pop("allowed_pairs") / max(1, stats.pop("density_den"))
    pk = peaks()
    # roofline of the kernel with the largest device time per step
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_step"])
    nl = kernels[dom]["launches_per_step"]
    km = {k: v / nl for k, v in kern.get(dom, {"flops": 0, "bytes": 0}).items()}
    kms = kernels[dom]["avg_ms"]
    t_tc = km.get("flops", 0) / (pk["bf16_tflops"] * 1e12)
    t_bw = km.get("bytes", 0) / (pk["hbm_gbs"] * 1e9)
    if t_tc >= t_bw:
        bound, achieved, peak, unit = "tensor", km["flops"] / kms / 1e9, pk["bf16_tflops"], "TFLOP/s"
    else:
        bound, achieved, peak, unit = "hbm", km["bytes"] / kms / 1e6, pk["hbm_gbs"], "GB/s"
    roof = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": profiled_traffic(dom, cfg.name),
            "peak_source": pk["source"] + " (burst)", "avg_launch_ms": kms, "launches_per_step": nl,
            "algorithmic_bytes_per_launch": km.get("bytes", 0),
            "algorithmic_flops_per_launch": km.get("flops", 0)}
    work = {}
    for k_ in ("annsa_tc", "annca_tc"):
        if k_ in kern and k_ in kernels and kern[k_].get("work_flops"):
            t_k = kernels[k_]["ms_per_step"]
            work[k_] = {"mma_flops_issued": kern[k_]["work_flops"], "algorithmic_flops": kern[k_]["flops"],
                        "TFLOP/s_issued": kern[k_]["work_flops"] / t_k / 1e9,
                        "frac_of_peak_issued": kern[k_]["work_flops"] / t_k / 1e9 / pk["bf16_tflops"],
                        "TFLOP/s_algorithmic": kern[k_]["flops"] / t_k / 1e9,
                        "GB/s_algorithmic": kern[k_]["bytes"] / t_k / 1e6,
                        "hbm_frac_algorithmic": kern[k_]["bytes"] / t_k / 1e6 / pk["hbm_gbs"],
                        # softmax exponentials: one per allowed (query, key)
                        # pair; at most one per tile element issued (32-key
                        # halves that no query of a warp meets are skipped)
                        "exp_algorithmic": kern[k_]["flops"] / (4 * cfg.D),
                        "exp_issued_at_most": kern[k_]["work_flops"] / (4 * cfg.D),
                        "exp_per_s_issued_at_most": kern[k_]["work_flops"] / (4 * cfg.D) / t_k * 1e3}
    kernel_roofs = {}
    for k_, m_ in kern.items():
        if k_ in kernels:
            t_k = kernels[k_]["ms_per_step"]
            kernel_roofs[k_] = {"GB/s": m_["bytes"] / t_k / 1e6, "hbm_frac": m_["bytes"] / t_k / 1e6 / pk["hbm_gbs"],
                                "TFLOP/s": m_["flops"] / t_k / 1e9,
                                "tensor_frac": m_["flops"] / t_k / 1e9 / pk["bf16_tflops"]}
    eff_tflops = sum(fl.values()) / ms / 1e9
    line = {"metric": METRIC, "value": value, "unit": "ms/chunk", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": value,
            "higher_is_better": False, "scaling": SCALING[args.shard], "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic (seeded; drawn on the GPU, see workloads/gen_device.py)"
            if cfg.prompt_clusters == 0 else "synthetic (seeded; host generator)",
            "config": config_dict(cfg, args, world),
            "rank0_share": {"layers": len(layers), "heads": len(heads)},
            "ms_median": ms_median,
            "l2_warm_ms": l2_warm,
            "effective_tflops": eff_tflops,
            "stages_ms": stage_ms,
            "roofline": roof,
            "attention_work_performed": work,
            "kernels": kernels,
            "kernel_rooflines": kernel_roofs,
            "stage_rooflines": {s_: {"GB/s": by[s_] / stage_ms[s_] / 1e6,
                                     "hbm_frac": by[s_] / stage_ms[s_] / 1e6 / pk["hbm_gbs"],
                                     "TFLOP/s": fl[s_] / stage_ms[s_] / 1e9} for s_ in stages},
            "work": stats,
            # the merge's kernels per layer: candidate set-up, per frame NN,
            # plan and apply, and the cache CSR (the other CSR is the query's)
            "merge_launches_per_layer": sum(kernels[k]["launches_per_step"] for k in
                                            ("cand_init", "cand_norm", "nn_tc", "plan", "apply")
                                            if k in kernels) / len(stack.paths) + 1,
            "gpu_launches": launches,
            "clocks": clk,
            "wall_s_timed": t_wall,
            "prep_s": t_prep,
            "e2e": {"value": e2e_ms, "unit": "ms/chunk", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "median": e2e_med, "min": e2e_min, "chunks": len(e2e)}}
    if cfg.P and sources[0].rel is not None:
        # AnnCA pruning of this chunk: kept prompt tokens per (head, frame)
        # and the share of the relevant tokens that survive
        p0 = stack.paths[0]
        kc = p0.kept_cnt.cpu().numpy()
        ki = p0.kept_idx.cpu().numpy()
        rel = np.asarray(sources[0].rel)
        hit = tot = 0
        for h in range(kc.shape[0]):
            for f in range(cfg.F):
                hit += int(rel[h][ki[h, f, :kc[h, f]]].sum())
                tot += int(rel[h].sum())
        line["prune"] = {"kept_per_head_frame": {"min": int(kc.min()), "mean": float(kc.mean()),
                                                 "max": int(kc.max()), "of": cfg.P},
                         "recall_relevant": hit / max(tot, 1), "relevant_share_of_prompt": float(rel.mean())}
    if want_dense:
        q, k, v, kp, vp = inputs[0]
        K, V = hist
        sd = dense_sdpa(q, K, V, kp, vp)
        line["dense"] = {"impl": "torch SDPA (bf16)", "keys": K.shape[1], "ms_per_layer": sd,
                         "ms": sd * cfg.layers, "timed": f"one layer of {len(heads)} heads, x {cfg.layers} layers",
                         "tflops": 4 * cfg.D * len(heads) * cfg.Nq * (K.shape[1] + cfg.P) / sd / 1e9}
        if cfg.D == 128:
            do = dense_ours(q, K, V, kp, vp, cfg.n_f, cfg.F)
            do["ms_per_layer"] = do["ms"]
            do["ms"] = do["ms"] * cfg.layers
            do["timed"] = f"one layer of {len(heads)} heads, x {cfg.layers} layers"
            line["dense_ours"] = do
        del K, V, hist
    del stack, inputs, snaps
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_rollout and cfg.idx == 4:
        line["rollout"] = rollout_measure(CONFIGS[2], args)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ob = oracle_baseline(cfg, 1, 0)
        line["cpu_baseline"] = {k: ob[k] for k in ("value", "unit", "cores", "kind", "sample", "unit_ms_mean",
                                                   "one_core_ms_per_chunk", "cpu_model", "host_cores",
                                                   "setup_s")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def recall_metrics(cfg, path, d, chunk_q, history_k=None, history_v=None):
    """Synthetic recall and density of one chunk's sparse selections, from
    the path's outputs: per head the share of the dense softmax mass that
    AnnSA's allowed slots carry (exp(lse of the kernel - dense lse), same
    logits: scale q.K + ln m over the live cache), the allowed density, the
    same share for AnnCA's kept prompt tokens, and, given the unmerged
    history, the relative error of the AnnSA output against dense attention
    over it.  Dense references are plain torch fp32 / SDPA (measurement)."""
    import torch
    import torch.nn.functional as Fn
    H, T = cfg.H, cfg.T
    q = torch.as_tensor(chunk_q).cuda().float()
    kp = torch.as_tensor(d.prompt_k).cuda().float()
    out = {"annsa_retained": [], "annsa_density": [], "annca_retained": [], "annca_kept_share": [],
           "annsa_rel_err_vs_dense_history": [], "annca_rel_err_vs_dense_prompt": [],
           "tempcache_rel_err_vs_dense_history": [], "tempcache_lse_gap": []}
    size = path.cache.size.tolist()
    lse = path.lse.float()
    for h in range(H):
        n = size[h]
        K = path.cache.K[h, :n].float()
        logits = cfg.scale * q[h] @ K.T + torch.log(path.cache.m[h, :n].float())[None, :]
        dense_lse = torch.logsumexp(logits, dim=1)
        out["annsa_retained"].append(float(torch.exp(lse[h] - dense_lse).mean()))
        allowed = torch.zeros_like(logits, dtype=torch.bool)
        for t in range(T):
            allowed |= path.q_codes[h, t][:, None] == path.cache.codes[h, t, :n][None, :]
        out["annsa_density"].append(float(allowed.float().mean()))
        if cfg.P:
            sp = torch.softmax(cfg.scale * q[h] @ kp[h].T, dim=1)
            ret, share = [], []
            for f in range(cfg.F):
                keep = torch.zeros(cfg.P, dtype=torch.bool, device="cuda")
                keep[path.kept_idx[h, f, :int(path.kept_cnt[h, f])].long()] = True
                ret.append(sp[f * cfg.n_f:(f + 1) * cfg.n_f][:, keep].sum(dim=1).mean())
                share.append(keep.float().mean())
            out["annca_retained"].append(float(torch.stack(ret).mean()))
            out["annca_kept_share"].append(float(torch.stack(share).mean()))
            o_ca_dense = Fn.scaled_dot_product_attention(q[h][None], kp[h][None],
                                                         torch.as_tensor(d.prompt_v[h]).cuda().float()[None])[0]
            out["annca_rel_err_vs_dense_prompt"].append(
                float((path.o_ca[h].float() - o_ca_dense).norm() / o_ca_dense.norm()))
        if history_k is not None:
            Kh = torch.as_tensor(history_k[h]).cuda().float()
            Vh = torch.as_tensor(history_v[h]).cuda().float()
            o_dense = Fn.scaled_dot_product_attention(q[h][None], Kh[None], Vh[None])[0]
            out["annsa_rel_err_vs_dense_history"].append(
                float((path.o_sa[h].float() - o_dense).norm() / o_dense.norm()))
            # TempCache alone: dense attention over the merged groups (+ ln m)
            # against dense attention over the unmerged history
            o_merged = torch.softmax(logits, dim=1) @ path.cache.V[h, :n].float()
            out["tempcache_rel_err_vs_dense_history"].append(
                float((o_merged - o_dense).norm() / o_dense.norm()))
            lse_hist = torch.logsumexp(cfg.scale * q[h] @ Kh.T, dim=1)
            out["tempcache_lse_gap"].append(float((dense_lse - lse_hist).abs().mean()))
    return {k: (float(np.mean(v)) if v else None) for k, v in out.items()}


def run_recall(args, cfg):
    """Sweep of the LSH and merge parameters on cfg's shapes (a seeded
    sample of heads): recall and density of AnnSA and AnnCA, and the output
    error against dense attention, per (tau, T, B)."""
    import torch

    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build as fbuild
    from merged_attention_autoregressive_gb300.path import ChunkPath

    fbuild.build()
    fa.lib()
    heads = [0, 5]
    # (tau, T, B, representative): the LSH / merge sweep with the method's
    # last-key groups, then the mean-key ablation (paperlayer.ai appendix C)
    settings = [(0.95, 2, 8, "last"), (0.90, 2, 8, "last"), (0.99, 2, 8, "last"), (0.95, 1, 8, "last"),
                (0.95, 4, 8, "last"), (0.95, 2, 6, "last"), (0.95, 2, 10, "last"),
                (0.95, 2, 8, "mean"), (0.90, 2, 8, "mean"), (0.99, 2, 8, "mean")]
    rows = []
    for tau, T, B, rep in settings:
        c = cfg.replace(H=len(heads), tau=tau, T=T, B=B)
        d = layer_data(c, chunks=1, heads=heads)
        todev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.bfloat16)  # noqa: E731
        path = ChunkPath(c.H, c.D, c.n_f, c.F, c.P, c.T, c.B, c.C, c.tau, torch.bfloat16, rep=rep)
        path.planes.copy_(todev(d.planes))
        f = 0
        while f < c.past_frames:
            nF = min(c.F, c.past_frames - f)
            path.merge(todev(np.concatenate(d.past_k[f:f + nF], 1)),
                       todev(np.concatenate(d.past_v[f:f + nF], 1)), f, F=nF)
            f += nF
        ins = [todev(x) for x in (d.chunk_q[0], d.chunk_k[0], d.chunk_v[0], d.prompt_k, d.prompt_v)]
        torch.cuda.synchronize()
        snap = path.cache.snapshot()
        # chunk latency on these heads (cache restored before each call, L2 warm)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ms = []
        for r in range(12):
            path.cache.restore(snap)
            ev[0].record()
            path.step(*ins, c.past_frames)
            ev[1].record()
            torch.cuda.synchronize()
            if r >= 2:
                ms.append(ev[0].elapsed_time(ev[1]))
        assert int(path.status.item()) == 0
        hk = np.concatenate(d.past_k + [d.chunk_k[0]], axis=1)
        hv = np.concatenate(d.past_v + [d.chunk_v[0]], axis=1)
        m = recall_metrics(c, path, d, d.chunk_q[0], hk, hv)
        m.update({"tau": tau, "T": T, "B": B, "rep": rep, "chunk_ms_2_heads_l2_warm": float(np.median(ms)),
                  "n_live_per_head": float(path.cache.size.float().mean()),
                  "keys_before_merge_per_head": (c.past_frames + c.F) * c.n_f})
        rows.append(m)
    line = {"metric": "synthetic recall / density of the sparse selections", "unit": "share",
            "data": "synthetic",
            "config": {"workload": cfg.name, "heads_sampled": heads, "D": cfg.D, "Nq": cfg.Nq,
                       "P": cfg.P, "past_frames": cfg.past_frames},
            "sweep": rows}
    print(json.dumps(line), flush=True)


def _slope_pct(ms):
    """Trend of a latency series in percent of its mean per 100 chunks (0
    for fewer than two chunks): the Theil-Sen estimate, the median of the
    slopes between every two chunks, so that a single slow chunk near either
    end of the window does not tilt it as it tilts a least-squares line."""
    y = np.asarray(ms, dtype=np.float64)
    if len(y) < 2:
        return 0.0
    i, j = np.triu_indices(len(y), 1)
    return float(np.median((y[j] - y[i]) / (j - i))) * 100.0 / float(y.mean()) * 100.0


def flatness(ms, resident, n_live=None, capacity=None):
    """Whether a rollout's per-chunk latency and memory stay flat.

    The trend is judged over the chunks at which the cache is full (n_live
    at capacity; at least 50 of them), else over the last 100 chunks: until
    the cache is full its live groups grow and the attention's cost with
    them, which is the expected fill, not growth of a full cache.  Flat =
    that trend under 1 % of the mean per 100 chunks, the 95th percentile of
    the last 50 chunks within 1.1 x their median (a percentile, so that one
    chunk's jitter on a sub-millisecond call does not decide it; the maximum
    is reported beside it) and the device bytes held identical at every
    chunk.  The trend of the last 100 chunks is reported either way."""
    ms = list(ms)
    slope100 = _slope_pct(ms[-100:])
    full = None
    if n_live is not None and capacity is not None:
        full = next((i for i, x in enumerate(n_live) if x >= capacity), None)
    steady = ms[full:] if full is not None and len(ms) - full >= 50 else None
    slope = _slope_pct(steady) if steady is not None else slope100
    last50 = np.array(ms[-50:], dtype=np.float64)
    med = float(np.median(last50))
    p95 = float(np.percentile(last50, 95))
    return {"ms_median_last50": med,
            "slope_last100_pct_of_mean_per_100_chunks": slope100,
            "slope_at_capacity_pct_of_mean_per_100_chunks": _slope_pct(steady) if steady is not None else None,
            "chunks_at_capacity": len(steady) if steady is not None else 0,
            "trend_window": "chunks at capacity" if steady is not None else "last 100 chunks",
            "max_over_median_last50": float(last50.max()) / med,
            "p95_over_median_last50": p95 / med,
            "flat": bool(abs(slope) < 1.0 and p95 <= 1.1 * med and min(resident) == max(resident))}


def rollout_measure(cfg, args):
    """A rollout of cfg.chunks chunks from an empty cache (the long-rollout
    workload, inputs drawn on the device): per chunk the latency of the
    public chunk call (L2 flushed before each), the live groups and the
    device memory held, and whether they stay flat.  Returns a dict."""
    import torch

    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300.path import ChunkPath
    from workloads.gen_device import DeviceLayerStream

    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    path = ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau, tdt, rep=args.rep)
    ds = DeviceLayerStream(cfg, 0)
    path.planes.copy_(ds.planes())
    kp, vp = ds.prompt()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    ms, n_live, resident = [], [], []
    n0 = fa.fastar_launch_count()
    t_wall = time.perf_counter()
    for c in range(cfg.chunks):
        fr = [ds.frame() for _ in range(cfg.F)]
        k, v, q = (torch.cat([f[i] for f in fr], dim=1).contiguous() for i in range(3))
        del fr
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        path.step(q, k, v, kp, vp, cfg.past_frames + c * cfg.F)
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
        n_live.append(float(path.cache.size.float().mean().item()))
        del q, k, v
        resident.append(torch.cuda.memory_allocated())
    t_wall = time.perf_counter() - t_wall
    assert int(path.status.item()) == 0, fa.STATUS.get(int(path.status.item()))
    launches = fa.fastar_launch_count() - n0
    row = cfg.D * 2 * (2 if cfg.dtype == "bf16" else 4)  # K and V bytes per key
    out = {"workload": cfg.name, "chunks": cfg.chunks, "H": cfg.H, "C": cfg.C,
           "ms_mean": float(np.mean(ms)), "ms_first_chunk": ms[0], "ms_median": float(np.median(ms)),
           **flatness(ms, resident, n_live, cfg.C),
           "ms_every_10th_chunk": ms[::10],
           "ms_last_100_chunks": [round(x, 5) for x in ms[-100:]],
           "n_live_every_10th_chunk": n_live[::10], "n_live_final": n_live[-1],
           "first_chunk_at_capacity": next((i for i, x in enumerate(n_live) if x >= cfg.C), None),
           "device_bytes_allocated": {"min": min(resident), "max": max(resident)},
           "cache_bytes": path.cache.nbytes(),
           "cache_live_kv_bytes_final": int(n_live[-1] * cfg.H * row),
           "dense_cache_keys_equiv": cfg.chunks * cfg.F * cfg.n_f,
           "dense_cache_kv_bytes_equiv": cfg.chunks * cfg.F * cfg.n_f * cfg.H * row,
           "gpu_launches": launches, "wall_s": t_wall,
           "l2": "flushed before every chunk (256 MiB write)",
           "data": "synthetic (seeded; drawn on the GPU)"}
    del path
    torch.cuda.empty_cache()
    return out


def run_rollout(args, cfg):
    """The long-rollout workload on its own (one JSON line)."""
    import torch

    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build as fbuild

    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    fbuild.build()
    fa.lib()
    clocks = Clocks(local)
    clocks.start()
    t0 = time.time()
    ro = rollout_measure(cfg, args)
    clocks.window(t0, time.time())
    clk = clocks.stop()
    line = {"metric": METRIC, "value": ro["ms_mean"], "unit": "ms/chunk", "n_gpus": 1,
            "steps": cfg.chunks, "warmup": 0, "ms_per_step": ro["ms_mean"],
            "higher_is_better": False, "scaling": "strong", "vs_baseline": None,
            "dtype": cfg.dtype, "data": ro["data"],
            "config": {"workload": cfg.name, "H": cfg.H, "D": cfg.D, "Nq": cfg.Nq, "P": cfg.P,
                       "T": cfg.T, "B": cfg.B, "C": cfg.C, "chunks": cfg.chunks, "l2": ro["l2"],
                       "parallelism": "single GPU"},
            "rollout": ro, "gpu_launches": ro["gpu_launches"], "clocks": clk}
    print(json.dumps(line), flush=True)


def run_quant(args, cfg):
    """The quantised matcher in place of the LSH buckets, per precision: one
    chunk of cfg's layer (past frames merged with the same search), the
    merge with TempCache-Quant, AnnCA-Quant and AnnSA-Quant one after the
    other on one stream (cache restored and L2 flushed before every rep),
    with k set to the pages' densities (AnnSA-Quant 28 %, AnnCA-Quant
    29.5 % of the keys); the share of the dense softmax mass each query
    keeps (same logits) and the density.  One JSON line."""
    import torch

    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build as fbuild
    from merged_attention_autoregressive_gb300.path import ChunkPath

    fbuild.build()
    fa.lib()
    bits_list = [int(b) for b in args.quant.split(",") if b]
    d = layer_data(cfg, chunks=1)
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.bfloat16)  # noqa: E731
    q, k, v = (todev(x) for x in (d.chunk_q[0], d.chunk_k[0], d.chunk_v[0]))
    kp, vp = todev(d.prompt_k), todev(d.prompt_v)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    rows = []
    for bits in bits_list:
        path = ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau, torch.bfloat16,
                         search=f"quant{bits}")
        path.planes.copy_(todev(d.planes))
        f = 0
        while f < cfg.past_frames:
            nF = min(cfg.F, cfg.past_frames - f)
            path.merge(todev(np.concatenate(d.past_k[f:f + nF], 1)), todev(np.concatenate(d.past_v[f:f + nF], 1)),
                       f, F=nF)
            f += nF
        torch.cuda.synchronize()
        snap = path.cache.snapshot()
        n_live = float(path.cache.size.float().mean())
        k_sa = max(1, int(round(0.28 * n_live)))
        k_ca = max(1, int(round(0.295 * cfg.P)))
        ws_sa = torch.empty(fa.fastar_workspace_size(fa.OP_QUANT, cfg.H, cfg.Nq, cfg.D, bits, 0, cfg.C),
                            dtype=torch.uint8, device="cuda")
        ws_ca = torch.empty(fa.fastar_workspace_size(fa.OP_QUANT, cfg.H, cfg.Nq, cfg.D, bits, 0, cfg.P),
                            dtype=torch.uint8, device="cuda")
        sel_ca = torch.zeros(cfg.H, cfg.Nq, (cfg.P + 31) // 32, dtype=torch.int32, device="cuda")
        st = path.status

        def chunk(ev=None):
            if ev:
                ev[0].record(stream)
            fa.fastar_hash(k, path.planes, cfg.T, cfg.B, path.k_codes, status=st)
            fa.fastar_tempcache_merge(path.cache, k, v, path.k_codes, cfg.F, cfg.n_f, cfg.past_frames, cfg.tau,
                                      match_out=path.match, ws=path.ws_merge, status=st, search=f"quant{bits}")
            if ev:
                ev[1].record(stream)
            fa.fastar_annca_quant_attention(q, kp, vp, path.scale, k_ca, bits, path.o_ca, sel_mask=sel_ca,
                                            ws=ws_ca, status=st)
            if ev:
                ev[2].record(stream)
            fa.fastar_annsa_quant_attention(q, path.cache, path.scale, k_sa, bits, path.o_sa, path.lse, ws=ws_sa,
                                            status=st)
            if ev:
                ev[3].record(stream)

        for _ in range(3):
            path.cache.restore(snap)
            chunk()
        reps = max(3, min(args.steps, 20))
        t = []
        for _ in range(reps):
            path.cache.restore(snap)
            flush.fill_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            chunk(ev)
            torch.cuda.synchronize()
            t.append([ev[i].elapsed_time(ev[i + 1]) for i in range(3)])
        assert int(st.item()) == 0, fa.STATUS.get(int(st.item()))
        t = np.median(np.array(t), axis=0)
        # recall: share of the dense softmax mass (same logits) each query keeps
        qf = q.float()
        sa_ret, ca_ret = [], []
        for h in range(cfg.H):
            n = int(path.cache.size[h])
            logits = path.scale * qf[h] @ path.cache.K[h, :n].float().T + torch.log(
                path.cache.m[h, :n].float())[None, :]
            sa_ret.append(float(torch.exp(path.lse[h] - torch.logsumexp(logits, dim=1)).mean()))
            sp = torch.softmax(path.scale * qf[h] @ kp[h].float().T, dim=1)
            m = sel_ca[h].long() & 0xFFFFFFFF
            bitsm = ((m[:, :, None] >> torch.arange(32, device="cuda")[None, None, :]) & 1).reshape(cfg.Nq, -1)
            ca_ret.append(float((sp * bitsm[:, :cfg.P].float()).sum(dim=1).mean()))
        rows.append({"bits": bits, "ms_merge": float(t[0]), "ms_annca_quant": float(t[1]),
                     "ms_annsa_quant": float(t[2]), "ms_chunk": float(t.sum()),
                     "n_live_per_head": n_live, "annsa_k": k_sa, "annsa_density": k_sa / n_live,
                     "annsa_retained": float(np.mean(sa_ret)), "annca_k": k_ca, "annca_density": k_ca / cfg.P,
                     "annca_retained": float(np.mean(ca_ret))})
        del path, ws_sa, ws_ca
        torch.cuda.empty_cache()
    line = {"metric": "per-chunk ms and retained softmax share of the quantised matcher", "unit": "ms/chunk",
            "value": rows[0]["ms_chunk"] if rows else None, "higher_is_better": False, "data": "synthetic",
            "config": {"workload": cfg.name, "H": cfg.H, "Nq": cfg.Nq, "P": cfg.P, "past_frames": cfg.past_frames,
                       "l2": "flushed before every chunk (256 MiB write)",
                       "k": "28 % of the live groups (AnnSA-Quant), 29.5 % of the prompt (AnnCA-Quant)"},
            "sweep": rows}
    print(json.dumps(line), flush=True)


def run_denoise(args, cfg):
    """The S denoising steps of one chunk on cfg's shapes (cache of the past
    frames built first): per chunk and per step device time with the
    pages' schedule (sparse attention off for the first 30 % of the steps),
    and with every step dense or every step sparse for comparison.  The
    cache is restored and L2 flushed before every chunk (untimed)."""
    import torch

    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build as fbuild
    from merged_attention_autoregressive_gb300.path import ChunkPath
    from workloads import denoise_steps

    fbuild.build()
    fa.lib()
    S = args.denoise
    d = layer_data(cfg, chunks=1)
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.bfloat16)  # noqa: E731
    path = ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau, torch.bfloat16)
    path.planes.copy_(todev(d.planes))
    f = 0
    while f < cfg.past_frames:
        nF = min(cfg.F, cfg.past_frames - f)
        path.merge(todev(np.concatenate(d.past_k[f:f + nF], 1)), todev(np.concatenate(d.past_v[f:f + nF], 1)),
                   f, F=nF)
        f += nF
    steps = [tuple(todev(x) for x in st) for st in denoise_steps(cfg, d, S)]
    kp, vp = todev(d.prompt_k), todev(d.prompt_v)
    torch.cuda.synchronize()
    snap = path.cache.snapshot()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def chunk(frac, ev=None, reuse=False, after=None):
        for s, (q, k, v) in enumerate(steps):
            path.denoise_step(s, S, q, k, v, kp, vp, cfg.past_frames, dense_frac=frac, reuse=reuse)
            if ev is not None:
                ev[s + 1].record(stream)
            if after is not None:
                after(s)

    heads = [0, 5]

    def retained(s):
        """Per step, on heads 0 and 5: the share of the dense softmax mass
        (same logits) that the step's selection keeps, exp(lse - dense lse);
        before the last step the dense set is the cache's groups (+ ln m)
        and the step's own keys, at the last step the merged cache."""
        q, k, _ = steps[s]
        out = []
        for h in heads:
            n = int(path.cache.size[h])
            logits = path.scale * q[h].float() @ path.cache.K[h, :n].float().T + torch.log(
                path.cache.m[h, :n].float())[None, :]
            if s + 1 < S:
                logits = torch.cat([logits, path.scale * q[h].float() @ k[h].float().T], dim=1)
            out.append(float(torch.exp(path.lse[h] - torch.logsumexp(logits, dim=1)).mean()))
        return float(np.mean(out))

    out = {}
    for name, frac, reuse in (("schedule_0.3", 0.3, False), ("schedule_0.3_reuse_codes", 0.3, True),
                              ("all_dense", 1.01, False), ("all_sparse", 0.0, False),
                              ("all_sparse_reuse_codes", 0.0, True)):
        for _ in range(3):
            path.cache.restore(snap)
            chunk(frac, reuse=reuse)
        reps = max(3, min(args.steps, 20))
        per_chunk, per_step = [], []
        for _ in range(reps):
            path.cache.restore(snap)
            flush.fill_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(S + 1)]
            ev[0].record(stream)
            chunk(frac, ev, reuse=reuse)
            torch.cuda.synchronize()
            per_chunk.append(ev[0].elapsed_time(ev[S]))
            per_step.append([ev[s].elapsed_time(ev[s + 1]) for s in range(S)])
        assert int(path.status.item()) == 0, fa.STATUS.get(int(path.status.item()))
        ret = []
        path.cache.restore(snap)
        chunk(frac, reuse=reuse, after=lambda s_: ret.append(retained(s_)))
        out[name] = {"ms_per_chunk": float(np.median(per_chunk)),
                     "ms_per_step": np.median(np.array(per_step), axis=0).round(4).tolist(),
                     "dense_steps": [s < frac * S for s in range(S)],
                     "retained_share_per_step_heads_0_5": [round(x, 5) for x in ret]}
    line = {"metric": "per-chunk FAST-AR attention ms over the denoising steps of a chunk", "unit": "ms/chunk",
            "value": out["schedule_0.3"]["ms_per_chunk"], "higher_is_better": False, "data": "synthetic",
            "config": {"workload": cfg.name, "H": cfg.H, "Nq": cfg.Nq, "P": cfg.P, "T": cfg.T, "B": cfg.B,
                       "past_frames": cfg.past_frames, "denoise_steps": S,
                       "l2": "flushed before every chunk (256 MiB write)",
                       "reuse_codes": "codes, query CSR and kept lists of the first sparse step reused by the "
                                      "later sparse steps (the last step re-hashes its keys for the merge)"},
            "schedules": out}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.config is None:
        args.config = 1 if (args.denoise or args.recall or args.quant) else 4
    cfg = CONFIGS[args.config]
    if args.layers:
        cfg = cfg.replace(layers=min(args.layers, cfg.layers))
    if args.impl == "reference":
        run_reference(args, cfg)
    elif args.quant:
        run_quant(args, cfg)
    elif args.denoise:
        run_denoise(args, cfg)
    elif args.recall:
        run_recall(args, cfg)
    elif cfg.chunks > 1:
        run_rollout(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
