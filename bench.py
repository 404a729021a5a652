#!/usr/bin/env python
"""Per-chunk FAST-AR attention path on one GB300: latency, TFLOP/s, roofline.

A step is one pass of the whole per-chunk path over one chunk of the
configured workload (default: one attention layer at Wan-1.3B-like width,
12 heads x D 128, 3 latent frames of 1560 tokens, 21 merged past frames,
512 prompt tokens, 2 LSH tables x 8 bits):
    hash(queries, new keys, prompt keys) -> TempCache merge (3 frames)
    -> AnnCA prune -> AnnCA attention -> AnnSA attention.
The timed step is the public per-chunk call (ChunkPath.step): the
cross-attention branch (prune, AnnCA) runs on a second stream beside the
merge and is joined before the call returns; CUDA events on the calling
stream bracket it.  The merge mutates the cache, so the pre-chunk cache
snapshot is restored before every step and L2 is flushed (a 256 MiB write)
outside the timed window.  Per-stage and per-kernel times come from
separate passes that run the stages one after the other on one stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `--impl reference` times the fp64 oracle on the
host cores instead (one head of the chunk per step, scaled to the chunk).
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--rep", default="last", choices=["last", "mean"],
                    help="TempCache representative: last key (the method) or mean key (ablation)")
    ap.add_argument("--denoise", type=int, default=0,
                    help="time the S denoising steps of one chunk (dense for the first 30%%) against "
                         "all-dense and all-sparse schedules (one JSON line)")
    ap.add_argument("--recall", action="store_true",
                    help="sweep tau, T and B: recall and density of AnnSA and AnnCA (one JSON line)")
    return ap.parse_args()


def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def rank_layer(rank: int) -> int:
    """The layer a rank runs: N GPUs run N independent layers of the same
    shape (weak scaling; heads and layers share nothing on the path)."""
    return rank


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
def oracle_chunk_one_head(cfg, d, head: int, st_head):
    """The oracle's whole per-chunk path for one head; returns seconds."""
    import oracle as O
    sl = slice(head, head + 1)
    q, k, v = d.chunk_q[0][sl], d.chunk_k[0][sl], d.chunk_v[0][sl]
    t0 = time.perf_counter()
    qc, _ = O.hash_codes(q, d.planes, cfg.T, cfg.B)
    O.bucket_csr(qc, 1 << cfg.B)
    kc, _ = O.hash_codes(k, d.planes, cfg.T, cfg.B)
    pc, _ = O.hash_codes(d.prompt_k[sl], d.planes, cfg.T, cfg.B)
    st, _, _ = O.tempcache_merge(st_head, k, v, kc, cfg.F, cfg.n_f, cfg.past_frames, cfg.tau)
    O.bucket_csr(st.codes, 1 << cfg.B)
    idx, cnt = O.annca_prune(qc, pc, cfg.F, cfg.n_f)
    O.annca_attention(q, d.prompt_k[sl], d.prompt_v[sl], idx, cnt, cfg.F, cfg.n_f, cfg.scale)
    O.annsa_attention(q, qc, st, cfg.scale)
    return time.perf_counter() - t0


def oracle_cache_one_head(cfg, d, head: int):
    import oracle as O
    sl = slice(head, head + 1)
    st = O.CacheState.empty(1, cfg.C, cfg.D, cfg.T, cfg.dtype)
    f = 0
    while f < cfg.past_frames:
        nF = min(cfg.F, cfg.past_frames - f)
        k = np.concatenate(d.past_k[f:f + nF], axis=1)[sl]
        v = np.concatenate(d.past_v[f:f + nF], axis=1)[sl]
        kc, _ = O.hash_codes(k, d.planes, cfg.T, cfg.B)
        st, _, _ = O.tempcache_merge(st, k, v, kc, nF, cfg.n_f, f, cfg.tau)
        f += nF
    return st


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, cfg):
    rank, world, _ = rank_info()
    if rank != 0:
        return
    d = layer_data(cfg, chunks=1)
    # one head of the chunk per step; the sample is capped at 24 heads so the
    # CPU run stays within a few minutes whatever --steps says
    n_meas = min(args.steps, 24)
    n_warm = min(args.warmup, 2)
    heads = [h % cfg.H for h in range(n_warm + n_meas)]
    states = {h: oracle_cache_one_head(cfg, d, h) for h in sorted(set(heads))}
    times = []
    for i, h in enumerate(heads):
        t = oracle_chunk_one_head(cfg, d, h, states[h])
        if i >= n_warm:
            times.append(t)
    per_chunk_ms = statistics.mean(times) * cfg.H * 1e3
    cores = host_cores()
    line = {"impl": "reference", "metric": METRIC, "value": per_chunk_ms, "unit": "ms/chunk",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_chunk_ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "H": cfg.H, "D": cfg.D, "Nq": cfg.Nq,
                       "P": cfg.P, "T": cfg.T, "B": cfg.B, "C": cfg.C},
            "cpu_baseline": {"value": per_chunk_ms, "unit": "ms/chunk", "cores": cores,
                             "kind": "oracle",
                             "sample": f"{n_meas} single-head samples of the {cfg.H}-head chunk "
                                       f"(heads in turn, after {n_warm} warm-up samples), mean x H; "
                                       "past frames merged untimed"},
            "e2e": {"value": per_chunk_ms, "unit": "ms/chunk", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU leg
def algorithmic(cfg, path, match, snap_size, snap_lf):
    """Algorithmic bytes and flops of one step, per stage and per kernel.

    Bytes count each input read once and each output written once; flops
    are 2*M*N*K for a GEMM and 4*D per (query, key) pair of attention.
    Returns (bytes per stage, flops per stage, per-kernel models, stats);
    a per-kernel model gives the bytes and flops of one launch (averaged over
    the launches of that kernel in a step).
    """
    import torch
    H, D, T, Nq, P, n_f, F = cfg.H, cfg.D, cfg.T, cfg.Nq, cfg.P, cfg.n_f, cfg.F
    e = 2 if cfg.dtype == "bf16" else 4
    size = path.cache.size.long()
    n_live = int(size.sum())
    kept = int(path.kept_cnt.long().sum())
    kept_tiles = int(((path.kept_cnt.long() + 63) // 64).sum())
    rows = H * (2 * Nq + P)
    by = {}
    by["hash"] = rows * (D * e + T * 4) + H * T * Nq * (4 + 4 + 4) + T * cfg.B * D * e
    # merge: new k, v read; candidate K read; matched V read; K, V written for
    # touched slots; per-slot metadata; cache CSR (codes read, perm written)
    mt = match.view(H, F, n_f)
    cand = []
    prev_cnt = int(((snap_lf == cfg.past_frames - 1) & (torch.arange(cfg.C, device=snap_lf.device)[None]
                                                         < snap_size[:, None])).sum())
    by["merge"] = 0
    for fi in range(F):
        cand.append(prev_cnt)
        m = mt[:, fi]
        n_matched = int((m >= 0).sum())
        n_groups = sum(int(torch.unique(m[h][m[h] >= 0]).numel()) for h in range(H))
        t_f = n_groups + int((m < 0).sum())
        prev_cnt = t_f
        by["merge"] += (2 * H * n_f * D * e + cand[-1] * D * e + n_matched * D * e
                        + 2 * t_f * D * e + t_f * (4 * 2 + T * 4) + H * n_f * 4 * 4)
    by["merge"] += n_live * T * (4 + 4) + H * T * ((1 << cfg.B) + 1) * 4
    by["prune"] = H * T * (Nq + P) * 4 + H * F * P * 4
    by["annca"] = H * Nq * D * e * 2 + kept * 2 * D * e + H * F * P * 4
    by["annsa"] = (H * Nq * D * e * 2 + H * T * Nq * 4 + n_live * (2 * D * e + 4 + 2 * T * 4)
                   + H * Nq * 4)
    # allowed pairs, split by the first table in which they collide
    pairs_t = [0] * T
    qc = path.q_codes.long()
    for h in range(H):
        n = int(size[h])
        cc = path.cache.codes[h, :, :n].long()
        for q0 in range(0, Nq, 1024):
            seen = torch.zeros(min(1024, Nq - q0), n, dtype=torch.bool, device=qc.device)
            for t in range(T):
                hit = (qc[h, t, q0:q0 + 1024, None] == cc[t][None]) & ~seen
                pairs_t[t] += int(hit.sum())
                seen |= hit
    pairs = sum(pairs_t)
    nn_flops = [2 * D * n_f * c for c in cand]
    fl = {"hash": 2 * rows * T * cfg.B * D, "merge": sum(nn_flops), "prune": 0,
          "annca": 4 * D * n_f * kept, "annsa": 4 * D * pairs}
    kern = {
        "nn_tc": {"flops": sum(nn_flops) / F,
                  "bytes": sum((H * n_f + c) * D * e for c in cand) / F},
        "annca_tc": {"flops": fl["annca"], "bytes": by["annca"]},
        # one launch for all tables; per table the queries and the live
        # slots (K, V, m, codes); with T > 1 each table writes an fp32
        # partial (o, max, sum) that the combine kernel reads back
        "annsa_tc": {"flops": fl["annsa"],
                     "bytes": (T * (H * Nq * D * e + n_live * (2 * D * e + 4 + 2 * T * 4))
                               + (T * H * Nq * (D * 4 + 8) if T > 1 else H * Nq * (D * e + 4)))},
        # the kept rows of each (head, frame), read once and written as
        # 64-row tiles (zero rows up to the tile) that annca_tc then loads
        "annca_compact": {"flops": 0, "bytes": 2 * kept * D * e + 2 * kept_tiles * 64 * D * e
                          + (kept + H * F) * 4},
        "annsa_combine": {"flops": 0, "bytes": T * H * Nq * (D * 4 + 8) + H * Nq * (D * e + 4)},
        # one launch for the queries, the new keys and the prompt keys
        "hash_tc": {"flops": 2 * rows * T * cfg.B * D, "bytes": rows * (D * e + T * 4)},
        "apply": {"flops": 0, "bytes": by["merge"] / F * 0.5},
    }
    return by, fl, kern, {"n_live": n_live, "kept": kept, "allowed_pairs": pairs,
                          "allowed_pairs_by_table": pairs_t,
                          "density": pairs / max(1, Nq * n_live)}


KERNEL_SOURCES = {"nn_tc": "nn_tc.cu", "annca_tc": "attention_tc.cu", "annsa_tc": "attention_tc.cu",
                  "hash_tc": "hash_tc.cu"}


def profiled_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic_<kernel>.txt), or None when there is none or the
    kernel's source has changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}.txt")
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


def dense_reference_ms(cfg, d, reps=10):
    """Dense attention of the same chunk: torch SDPA over the unmerged history."""
    import torch
    import torch.nn.functional as Fn
    dt = torch.bfloat16
    K = torch.from_numpy(np.concatenate(d.past_k + [d.chunk_k[0]], axis=1)).to("cuda", dt)
    V = torch.from_numpy(np.concatenate(d.past_v + [d.chunk_v[0]], axis=1)).to("cuda", dt)
    q = torch.from_numpy(d.chunk_q[0]).to("cuda", dt)
    kp = torch.from_numpy(d.prompt_k).to("cuda", dt)
    vp = torch.from_numpy(d.prompt_v).to("cuda", dt)

    def run():
        Fn.scaled_dot_product_attention(q[None], K[None], V[None])
        Fn.scaled_dot_product_attention(q[None], kp[None], vp[None])
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        run()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / reps
    n_keys = K.shape[1]
    flops = 4 * cfg.D * cfg.H * cfg.Nq * (n_keys + cfg.P)
    return {"ms": ms, "keys": n_keys, "tflops": flops / ms / 1e9, "impl": "torch SDPA (bf16)"}


def dense_ours(cfg, d, reps=10):
    """Dense attention of the same chunk through this library's own kernels.

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
    dt = torch.bfloat16
    H, D, Nq, P, F = cfg.H, cfg.D, cfg.Nq, cfg.P, cfg.F
    K = torch.from_numpy(np.concatenate(d.past_k + [d.chunk_k[0]], axis=1)).to("cuda", dt)
    V = torch.from_numpy(np.concatenate(d.past_v + [d.chunk_v[0]], axis=1)).to("cuda", dt)
    n = K.shape[1]
    q = torch.from_numpy(d.chunk_q[0]).to("cuda", dt)
    kp = torch.from_numpy(d.prompt_k).to("cuda", dt)
    vp = torch.from_numpy(d.prompt_v).to("cuda", dt)
    c = fa.Cache(H, n, D, 1, 1, dt)
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
    o_sa = torch.empty(H, Nq, D, dtype=dt, device="cuda")
    o_ca = torch.empty(H, Nq, D, dtype=dt, device="cuda")
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
            fa.fastar_annca_attention(q, kp, vp, kept_idx, kept_cnt, F, cfg.n_f, scale, o_ca, ws=ws_ca,
                                      status=st)

    def timed(fn):
        for _ in range(3):
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
    del c, K, V
    torch.cuda.empty_cache()
    return out


def run_ours(args, cfg):
    import torch
    import torch.distributed as dist

    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build as fbuild
    from merged_attention_autoregressive_gb300.path import ChunkPath

    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fbuild.build()
    fa.lib()
    d = layer_data(cfg, layer=rank_layer(rank), chunks=1)
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", tdt)  # noqa: E731
    path = ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau, tdt, rep=args.rep)
    path.planes.copy_(todev(d.planes))
    f = 0
    while f < cfg.past_frames:
        nF = min(cfg.F, cfg.past_frames - f)
        path.merge(todev(np.concatenate(d.past_k[f:f + nF], 1)),
                   todev(np.concatenate(d.past_v[f:f + nF], 1)), f, F=nF)
        f += nF
    torch.cuda.synchronize()
    snap = path.cache.snapshot()
    q, k, v = todev(d.chunk_q[0]), todev(d.chunk_k[0]), todev(d.chunk_v[0])
    kp, vp = todev(d.prompt_k), todev(d.prompt_v)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    first = cfg.past_frames
    st = path.status
    stages = ["hash", "merge", "prune", "annca", "annsa"]

    def step(ev=None):
        rec = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
        rec(0)
        fa.fastar_hash_many([(q, path.q_codes, path.q_perm, path.q_offsets),
                             (k, path.k_codes, None, None), (kp, path.p_codes, None, None)],
                            path.planes, cfg.T, cfg.B, status=st)
        rec(1)
        fa.fastar_tempcache_merge(path.cache, k, v, path.k_codes, cfg.F, cfg.n_f, first, cfg.tau,
                                  match_out=path.match, ws=path.ws_merge, status=st, rep=args.rep,
                                  planes=path.planes)
        rec(2)
        fa.fastar_annca_prune(path.q_codes, path.p_codes, cfg.F, cfg.n_f, cfg.B, path.kept_idx,
                              path.kept_cnt, status=st)
        rec(3)
        fa.fastar_annca_attention(q, kp, vp, path.kept_idx, path.kept_cnt, cfg.F, cfg.n_f,
                                  path.scale, path.o_ca, ws=path.ws_annca, status=st)
        rec(4)
        fa.fastar_annsa_attention(q, path.q_codes, path.q_perm, path.q_offsets, path.cache,
                                  path.scale, path.o_sa, path.lse, ws=path.ws_annsa, status=st)
        rec(5)

    def chunk():
        # the public per-chunk call: the cross-attention branch runs on a
        # second stream and is joined before it returns
        path.step(q, k, v, kp, vp, first)

    def prep():
        path.cache.restore(snap)
        flush.fill_(1)

    for _ in range(max(3, args.warmup)):
        prep()
        chunk()
        prep()
        step()
    torch.cuda.synchronize()
    assert int(st.item()) == 0, fa.STATUS.get(int(st.item()))
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
        chunk()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks.window(t0, time.time())
    clk = clocks.stop()
    launches = fa.fastar_launch_count() - n0
    assert int(st.item()) == 0, fa.STATUS.get(int(st.item()))
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms = statistics.mean(step_ms)
    # per-stage times: a separate pass that runs the stages one after the
    # other on one stream, with events between them
    n_ssteps = min(args.steps, 50)
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_ssteps)]
    for i in range(n_ssteps):
        prep()
        step(sevs[i])
    torch.cuda.synchronize()
    stage_ms = {s: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in sevs)
                for j, s in enumerate(stages)}
    # the job's time is its slowest rank's; every rank ran args.steps chunks
    total_ms = job_max(sum(step_ms), world, "cuda")
    value = total_ms / (args.steps * world)

    # per-kernel durations: a separate pass with the library's launch timer
    # (same restore + L2 flush protocol), events on the launch stream
    timer = fa.LaunchTimer(64)
    per_kernel = {}
    n_tsteps = min(args.steps, 50)
    for i in range(n_tsteps):
        prep()
        timer.begin()
        step()
        for name, ms_k in timer.end():
            per_kernel.setdefault(name, []).append(ms_k)
    kernels = {k: {"launches_per_step": len(v) / n_tsteps, "avg_ms": statistics.mean(v),
                   "ms_per_step": sum(v) / n_tsteps} for k, v in per_kernel.items()}

    # end to end through the C ABI with host buffers (pinned), copies timed
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
    hkp, hvp = kp.cpu().pin_memory(), vp.cpu().pin_memory()
    ho_ca, ho_sa = torch.empty_like(path.o_ca, device="cpu").pin_memory(), \
        torch.empty_like(path.o_sa, device="cpu").pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hkp, hvp))
    d2h = ho_ca.numel() * ho_ca.element_size() + ho_sa.numel() * ho_sa.element_size()
    e2e = []
    for i in range(args.steps + 3):
        prep()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        # the public host-to-host chunk: copies in per branch, outputs copied
        # out as soon as they are final, all inside the timed region
        path.step_host(hq, hk, hv, hkp, hvp, ho_ca, ho_sa, first)
        s1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            e2e.append(s0.elapsed_time(s1))
    e2e_ms = statistics.mean(e2e)

    # algorithmic work of the step (from the last step's outputs)
    by, fl, kern, stats = algorithmic(cfg, path, path.match.clone(), snap["size"], snap["last_frame"])
    pk = peaks()
    # roofline of the kernel with the largest device time per step
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_step"])
    km = kern.get(dom, {"flops": 0, "bytes": 0})
    kms = kernels[dom]["avg_ms"]
    t_tc = km["flops"] / (pk["bf16_tflops"] * 1e12)
    t_bw = km["bytes"] / (pk["hbm_gbs"] * 1e9)
    if t_tc >= t_bw:
        bound, achieved, peak, unit = "tensor", km["flops"] / kms / 1e9, pk["bf16_tflops"], "TFLOP/s"
    else:
        bound, achieved, peak, unit = "hbm", km["bytes"] / kms / 1e6, pk["hbm_gbs"], "GB/s"
    traffic = profiled_traffic(dom)
    eff_tflops = sum(fl.values()) / ms / 1e9
    line = {"metric": METRIC, "value": value, "unit": "ms/chunk", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": cfg.name, "H": cfg.H, "D": cfg.D, "Nq": cfg.Nq, "P": cfg.P,
                       "T": cfg.T, "B": cfg.B, "C": cfg.C, "past_frames": cfg.past_frames,
                       "l2": "flushed before every step (256 MiB write)", "representative": args.rep,
                       "parallelism": (f"layer-parallel x{world}: rank r runs layer r, no collective"
                                       if world > 1 else "single GPU")},
            "effective_tflops": eff_tflops,
            "stages_ms": stage_ms,
            "roofline": {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak,
                         "unit": unit, "frac": achieved / peak, "traffic": traffic,
                         "peak_source": pk["source"] + " (burst)",
                         "avg_launch_ms": kms, "launches_per_step": kernels[dom]["launches_per_step"],
                         "algorithmic_bytes_per_launch": km["bytes"],
                         "algorithmic_flops_per_launch": km["flops"]},
            "kernels": kernels,
            "stage_rooflines": {s: {"GB/s": by[s] / stage_ms[s] / 1e6,
                                    "hbm_frac": by[s] / stage_ms[s] / 1e6 / pk["hbm_gbs"],
                                    "TFLOP/s": fl[s] / stage_ms[s] / 1e9} for s in stages},
            "work": stats,
            "gpu_launches": launches,
            "clocks": clk,
            "wall_s_timed": t_wall,
            "e2e": {"value": e2e_ms, "unit": "ms/chunk", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h}}
    if cfg.P:
        # AnnCA pruning of this chunk: kept prompt tokens per (head, frame)
        # and, where the prompt has a relevance label, the share of the
        # relevant tokens that survive
        kc = path.kept_cnt.cpu().numpy()
        ki = path.kept_idx.cpu().numpy()
        rel = np.asarray(d.prompt_rel)
        pr = {"kept_per_head_frame": {"min": int(kc.min()), "mean": float(kc.mean()),
                                      "max": int(kc.max()), "of": cfg.P}}
        if not rel.all():
            hit = tot = 0
            for h in range(cfg.H):
                for f in range(cfg.F):
                    kept = ki[h, f, :kc[h, f]]
                    hit += int(rel[h][kept].sum())
                    tot += int(rel[h].sum())
            pr["recall_relevant"] = hit / max(tot, 1)
            pr["relevant_share_of_prompt"] = float(rel.mean())
        line["prune"] = pr
    if cfg.layers > 1:
        # layers are independent and identical in shape: one layer is timed
        # and the per-chunk figures are scaled to all of them
        L = cfg.layers
        line["value"] *= L
        line["ms_per_step"] *= L
        line["e2e"]["value"] *= L
        line["e2e"]["h2d_bytes_per_step"] *= L
        line["e2e"]["d2h_bytes_per_step"] *= L
        line["config"]["layers"] = L
        line["config"]["timed_layers"] = 1
        line["config"]["scaled"] = f"one layer timed, x{L}"
    if not args.no_dense and rank == 0:
        line["dense"] = dense_reference_ms(cfg, d)
        if cfg.layers > 1:
            line["dense"]["ms_all_layers"] = line["dense"]["ms"] * cfg.layers
        if cfg.dtype == "bf16" and cfg.D == 128:
            line["dense_ours"] = dense_ours(cfg, d)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        h = 0
        st_h = oracle_cache_one_head(cfg, d, h)
        secs = [oracle_chunk_one_head(cfg, d, h, st_h) for _ in range(2)]
        line["cpu_baseline"] = {"value": min(secs) * cfg.H * 1e3, "unit": "ms/chunk",
                                "cores": host_cores(), "kind": "oracle",
                                "sample": "head 0 of the chunk (best of 2), x H heads"}
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


def run_rollout(args, cfg):
    """A rollout of cfg.chunks chunks from an empty cache (the long-rollout
    workload): per chunk the latency of the public chunk call, the live
    groups and the device memory held, and whether they stay flat."""
    import torch

    import merged_attention_autoregressive_gb300 as fa
    from merged_attention_autoregressive_gb300 import build as fbuild
    from merged_attention_autoregressive_gb300.path import ChunkPath
    from workloads.gen import HeadStream, planes as gen_planes, prompt as gen_prompt

    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    fbuild.build()
    fa.lib()
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    todev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", tdt)  # noqa: E731
    path = ChunkPath(cfg.H, cfg.D, cfg.n_f, cfg.F, cfg.P, cfg.T, cfg.B, cfg.C, cfg.tau, tdt)
    path.planes.copy_(todev(gen_planes(cfg, 0)))
    streams = [HeadStream(cfg, 0, h) for h in range(cfg.H)]
    pk, pv, _ = zip(*[gen_prompt(cfg, 0, h, s.centroids) for h, s in enumerate(streams)])
    kp, vp = todev(np.stack(pk)), todev(np.stack(pv))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def next_chunk():
        fr = [[s.frame() for _ in range(cfg.F)] for s in streams]
        cat = lambda i: todev(np.stack([np.concatenate([f[i] for f in hf], axis=0) for hf in fr]))  # noqa: E731
        return cat(2), cat(0), cat(1)  # q, k, v

    ms, n_live, resident = [], [], []
    n0 = fa.fastar_launch_count()
    clocks = Clocks(local)
    clocks.start()
    t0 = time.time()
    for c in range(cfg.chunks):
        q, k, v = next_chunk()
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        path.step(q, k, v, kp, vp, cfg.past_frames + c * cfg.F)
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
        n_live.append(float(path.cache.size.float().mean().item()))
        resident.append(torch.cuda.memory_allocated())
    clocks.window(t0, time.time())
    clk = clocks.stop()
    assert int(path.status.item()) == 0, fa.STATUS.get(int(path.status.item()))
    launches = fa.fastar_launch_count() - n0
    tail = np.array(ms[-100:]) if len(ms) >= 100 else np.array(ms)
    slope = float(np.polyfit(np.arange(len(tail)), tail, 1)[0]) * 100 / float(tail.mean())
    last50 = np.array(ms[-50:])
    row = cfg.D * 2 * (2 if cfg.dtype == "bf16" else 4)  # K and V bytes per key
    line = {"metric": METRIC, "value": float(np.mean(ms)), "unit": "ms/chunk", "n_gpus": 1,
            "steps": cfg.chunks, "warmup": 0, "ms_per_step": float(np.mean(ms)),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": cfg.name, "H": cfg.H, "D": cfg.D, "Nq": cfg.Nq, "P": cfg.P,
                       "T": cfg.T, "B": cfg.B, "C": cfg.C, "chunks": cfg.chunks,
                       "l2": "flushed before every chunk (256 MiB write)",
                       "parallelism": "single GPU"},
            "rollout": {
                "ms_first_chunk": ms[0], "ms_median": float(np.median(ms)),
                "ms_median_last50": float(np.median(last50)),
                "slope_last100_pct_of_mean_per_100_chunks": slope,
                "max_over_median_last50": float(last50.max() / np.median(last50)),
                "ms_every_10th_chunk": ms[::10],
                "n_live_every_10th_chunk": n_live[::10], "n_live_final": n_live[-1],
                "device_bytes_allocated": {"min": min(resident), "max": max(resident)},
                "cache_live_kv_bytes_final": int(n_live[-1] * cfg.H * row),
                "dense_cache_keys_equiv": cfg.chunks * cfg.F * cfg.n_f,
                "dense_cache_kv_bytes_equiv": cfg.chunks * cfg.F * cfg.n_f * cfg.H * row},
            "gpu_launches": launches, "clocks": clk}
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

    def chunk(frac, ev=None):
        for s, (q, k, v) in enumerate(steps):
            path.denoise_step(s, S, q, k, v, kp, vp, cfg.past_frames, dense_frac=frac)
            if ev is not None:
                ev[s + 1].record(stream)

    out = {}
    for name, frac in (("schedule_0.3", 0.3), ("all_dense", 1.01), ("all_sparse", 0.0)):
        for _ in range(3):
            path.cache.restore(snap)
            chunk(frac)
        reps = max(3, min(args.steps, 20))
        per_chunk, per_step = [], []
        for _ in range(reps):
            path.cache.restore(snap)
            flush.fill_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(S + 1)]
            ev[0].record(stream)
            chunk(frac, ev)
            torch.cuda.synchronize()
            per_chunk.append(ev[0].elapsed_time(ev[S]))
            per_step.append([ev[s].elapsed_time(ev[s + 1]) for s in range(S)])
        assert int(path.status.item()) == 0, fa.STATUS.get(int(path.status.item()))
        out[name] = {"ms_per_chunk": float(np.median(per_chunk)),
                     "ms_per_step": np.median(np.array(per_step), axis=0).round(4).tolist(),
                     "dense_steps": [s < frac * S for s in range(S)]}
    line = {"metric": "per-chunk FAST-AR attention ms over the denoising steps of a chunk", "unit": "ms/chunk",
            "value": out["schedule_0.3"]["ms_per_chunk"], "higher_is_better": False, "data": "synthetic",
            "config": {"workload": cfg.name, "H": cfg.H, "Nq": cfg.Nq, "P": cfg.P, "T": cfg.T, "B": cfg.B,
                       "past_frames": cfg.past_frames, "denoise_steps": S,
                       "l2": "flushed before every chunk (256 MiB write)"},
            "schedules": out}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg)
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
