"""Seeded synthetic inputs for the FAST-AR per-chunk attention path.

This module only draws random numbers and rounds them to the storage type;
it holds none of the method's arithmetic, so both the fp64 oracle and the
CUDA library consume exactly the same bits from it.

What the pages describe, and what the synthetic data imitates
-------------------------------------------------------------
* Keys and queries are strongly semantic: they form clusters (foreground
  and background objects) -- FAST-AR summary (paperlayer.ai), section 4
  "Motivation", self-attention redundancy bullet; FAST-AR analysis
  (paper.rainbus.top), figure 3 description.
* Cached keys repeat across frames (near-duplicates) -- same passages, and
  the abstract, which names cached keys that nearly repeat frame to frame.
* Each prompt only matters for a few tokens per frame -- paperlayer.ai,
  section 4, cross-attention overhead bullet; rainbus figure 4.

Recipe (one independent stream per (config, layer, head, purpose)):
  * cluster centroids: unit-norm Gaussian directions;
  * frame 0 keys: centroid of a uniformly drawn cluster + N(0, sigma^2 I)
    per coordinate (sigma = 0.1);
  * frame f keys: a random permutation of frame f-1's keys plus
    N(0, 0.02^2 I) per coordinate; a fraction `redraw` of positions is then
    redrawn fresh from the mixture (new cluster, new key);
  * values: i.i.d. N(0, 1), fresh for every token of every frame;
  * query i of frame f: centroid of key i's cluster + fresh N(0, sigma^2 I);
  * prompt keys: from the same mixture as the keys (long-prompt config:
    256 prompt clusters, 16 of which are query clusters);
  * LSH hyperplanes: N(0, 1), one set [T*B][D] per layer, shared by all
    heads and by queries, keys and prompt keys.
Every array is drawn in float32 and rounded once, round-to-nearest-even,
to bf16 (bf16 configs) and returned as float32 arrays holding exactly
bf16-representable values.

These stand in for the pages' benchmarks (LongVBench, LongVGenBench) and
for model activations, which are not available here.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

ROOT_SEED = 20260202

# purposes of the per-(config, layer, head) streams
_P_CENTROIDS, _P_KEYS, _P_VALUES, _P_QUERIES, _P_PROMPT, _P_PROMPT_V = 0, 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Config:
    """Shapes and data recipe of one workload."""
    idx: int
    name: str
    H: int              # heads
    D: int              # head dim
    dtype: str          # "bf16" or "f32" (storage and kernel input type)
    n_f: int            # tokens per latent frame
    F: int              # frames per chunk
    past_frames: int    # frames merged into the cache before the measured chunk
    P: int              # prompt tokens
    T: int              # LSH tables
    B: int              # bits per table
    tau: float          # TempCache cosine threshold
    C: int              # cache capacity per head
    clusters: int       # key/query clusters per head
    sigma: float = 0.1
    frame_noise: float = 0.02
    redraw: float = 0.10
    chunks: int = 1     # chunks generated after the past frames
    layers: int = 1     # independent layers per chunk
    prompt_clusters: int = 0   # long-prompt config: clusters of the prompt
    prompt_overlap: int = 0    # ... of which this many are query clusters

    @property
    def Nq(self) -> int:
        return self.F * self.n_f

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS = [
    # tiny fp32 check: 4 past frames x 256 + one 256-token frame, prompt 64
    Config(0, "tiny_fp32_h1_d64", H=1, D=64, dtype="f32", n_f=256, F=1,
           past_frames=4, P=64, T=1, B=6, tau=0.95, C=1024, clusters=8,
           redraw=0.20),
    # one attention layer at Wan-1.3B-like width (bench workload)
    Config(1, "wan1.3b_layer_h12_d128", H=12, D=128, dtype="bf16", n_f=1560,
           F=3, past_frames=21, P=512, T=2, B=8, tau=0.95, C=32768,
           clusters=64, redraw=0.10),
    # 200-chunk rollout with the same shapes
    Config(2, "rollout200_h12_d128", H=12, D=128, dtype="bf16", n_f=1560,
           F=3, past_frames=0, P=512, T=2, B=8, tau=0.95, C=32768,
           clusters=64, redraw=0.05, chunks=200),
    # long-prompt cross-attention stress
    Config(3, "long_prompt_ca_h12_d128", H=12, D=128, dtype="bf16",
           n_f=1560, F=3, past_frames=0, P=4096, T=4, B=10, tau=0.95,
           C=32768, clusters=64, redraw=0.10, prompt_clusters=256,
           prompt_overlap=16),
    # 14B-like 720p chunk, 40 independent layers
    Config(4, "14b_720p_h40_d128", H=40, D=128, dtype="bf16", n_f=3600, F=3,
           past_frames=21, P=512, T=2, B=10, tau=0.95, C=32768,
           clusters=128, redraw=0.10, layers=40),
]


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(dtype)


def _rng(cfg: Config, layer: int, head: int, purpose: int, extra: int = 0):
    ss = np.random.SeedSequence([ROOT_SEED, cfg.idx, layer, head, purpose, extra])
    return np.random.Generator(np.random.PCG64(ss))


def _unit_rows(rng, n, d):
    c = rng.standard_normal((n, d), dtype=np.float32)
    c /= np.linalg.norm(c, axis=1, keepdims=True)
    return c


def planes(cfg: Config, layer: int = 0) -> np.ndarray:
    """LSH hyperplanes [T*B][D], N(0,1), rounded to the storage type."""
    rng = _rng(cfg, layer, 0xFFFF, 9)
    r = rng.standard_normal((cfg.T * cfg.B, cfg.D), dtype=np.float32)
    return to_storage(r, cfg.dtype)


class HeadStream:
    """Frame-by-frame keys, values and queries of one (layer, head).

    Frames must be requested in order 0, 1, 2, ... (the key process is a
    Markov chain over frames).
    """

    def __init__(self, cfg: Config, layer: int, head: int):
        self.cfg, self.layer, self.head = cfg, layer, head
        self.centroids = _unit_rows(_rng(cfg, layer, head, _P_CENTROIDS),
                                    cfg.clusters, cfg.D)
        self._rk = _rng(cfg, layer, head, _P_KEYS)
        self._rv = _rng(cfg, layer, head, _P_VALUES)
        self._rq = _rng(cfg, layer, head, _P_QUERIES)
        self.next_frame = 0
        self._keys = None       # storage-rounded keys of the last frame
        self._clus = None       # their cluster ids

    def _fresh(self, n):
        c = self._rk.integers(0, self.cfg.clusters, size=n)
        x = self.centroids[c] + self.cfg.sigma * self._rk.standard_normal(
            (n, self.cfg.D), dtype=np.float32)
        return c, x

    def frame(self):
        """Return (keys, values, queries, clusters) of the next frame."""
        cfg = self.cfg
        n, D = cfg.n_f, cfg.D
        if self._keys is None:
            clus, k = self._fresh(n)
        else:
            perm = self._rk.permutation(n)
            k = self._keys[perm] + cfg.frame_noise * self._rk.standard_normal(
                (n, D), dtype=np.float32)
            clus = self._clus[perm].copy()
            nred = int(round(cfg.redraw * n))
            if nred:
                pos = self._rk.choice(n, size=nred, replace=False)
                c2, k2 = self._fresh(nred)
                k[pos] = k2
                clus[pos] = c2
        k = to_storage(k, cfg.dtype)
        v = to_storage(self._rv.standard_normal((n, D), dtype=np.float32), cfg.dtype)
        q = self.centroids[clus] + cfg.sigma * self._rq.standard_normal(
            (n, D), dtype=np.float32)
        q = to_storage(q, cfg.dtype)
        self._keys, self._clus = k, clus
        self.next_frame += 1
        return k, v, q, clus


def prompt(cfg: Config, layer: int, head: int, centroids: np.ndarray):
    """Prompt keys [P][D], values [P][D] and a relevance label [P] (bool).

    The label marks tokens drawn from a cluster that the queries also use
    (always true when the prompt shares the key mixture).
    """
    rng = _rng(cfg, layer, head, _P_PROMPT)
    P, D = cfg.P, cfg.D
    if cfg.prompt_clusters:
        pc = _unit_rows(rng, cfg.prompt_clusters, D)
        shared = rng.choice(cfg.clusters, size=cfg.prompt_overlap, replace=False)
        pc[: cfg.prompt_overlap] = centroids[shared]
        c = rng.integers(0, cfg.prompt_clusters, size=P)
        k = pc[c] + cfg.sigma * rng.standard_normal((P, D), dtype=np.float32)
        rel = c < cfg.prompt_overlap
    else:
        c = rng.integers(0, cfg.clusters, size=P)
        k = centroids[c] + cfg.sigma * rng.standard_normal((P, D), dtype=np.float32)
        rel = np.ones(P, dtype=bool)
    v = _rng(cfg, layer, head, _P_PROMPT_V).standard_normal((P, D), dtype=np.float32)
    return to_storage(k, cfg.dtype), to_storage(v, cfg.dtype), rel


@dataclass
class LayerData:
    """All inputs of one layer: past frames, the chunks after them, prompt.

    Arrays are stacked over heads: past_k[frame] has shape [H][n_f][D],
    chunk_k[chunk] has shape [H][F*n_f][D].
    """
    cfg: Config
    layer: int
    planes: np.ndarray          # [T*B][D]
    past_k: list                # past_frames x [H][n_f][D]
    past_v: list
    chunk_k: list               # chunks x [H][F*n_f][D]
    chunk_v: list
    chunk_q: list
    prompt_k: np.ndarray        # [H][P][D]
    prompt_v: np.ndarray
    prompt_rel: np.ndarray      # [H][P] bool


def layer_data(cfg: Config, layer: int = 0, chunks: int | None = None,
               heads=None) -> LayerData:
    """Generate past frames, `chunks` chunks and the prompt for one layer."""
    chunks = cfg.chunks if chunks is None else chunks
    heads = list(range(cfg.H)) if heads is None else list(heads)
    streams = [HeadStream(cfg, layer, h) for h in heads]
    past_k, past_v = [], []
    for _ in range(cfg.past_frames):
        fr = [s.frame() for s in streams]
        past_k.append(np.stack([f[0] for f in fr]))
        past_v.append(np.stack([f[1] for f in fr]))
    ck, cv, cq = [], [], []
    for _ in range(chunks):
        ks, vs, qs = [], [], []
        for _f in range(cfg.F):
            fr = [s.frame() for s in streams]
            ks.append(np.stack([f[0] for f in fr]))
            vs.append(np.stack([f[1] for f in fr]))
            qs.append(np.stack([f[2] for f in fr]))
        ck.append(np.concatenate(ks, axis=1))
        cv.append(np.concatenate(vs, axis=1))
        cq.append(np.concatenate(qs, axis=1))
    pk, pv, pr = zip(*[prompt(cfg, layer, h, s.centroids) for h, s in zip(heads, streams)])
    return LayerData(cfg, layer, planes(cfg, layer), past_k, past_v, ck, cv, cq,
                     np.stack(pk), np.stack(pv), np.stack(pr))


_P_DENOISE = 6


def denoise_steps(cfg: Config, d: LayerData, S: int, chunk: int = 0, layer: int = 0):
    """Inputs of the S denoising steps of chunk `chunk`: step s sees the
    chunk's queries, keys and values plus N(0, sigma_s^2) per coordinate,
    sigma_s = 0.05 (S - 1 - s) (the last step sees the clean chunk), each
    drawn from its own stream and rounded once to the storage type.  A
    stand-in for the activations of successive denoising steps, which change
    less as the latent gets cleaner."""
    out = []
    for s in range(S):
        sigma = 0.05 * (S - 1 - s)
        rng = _rng(cfg, layer, 0, _P_DENOISE, extra=chunk * 1000 + s)
        step = []
        for x in (d.chunk_q[chunk], d.chunk_k[chunk], d.chunk_v[chunk]):
            noise = rng.standard_normal(x.shape, dtype=np.float32) * np.float32(sigma)
            step.append(to_storage(x + noise, cfg.dtype))
        out.append(tuple(step))
    return out
