"""Seeded synthetic inputs drawn on the GPU, for workloads too large to draw
on the host in reasonable time (the 40-layer 14B-like chunk).

The recipe is the one of workloads/gen.py, drawn with torch's device
generator instead of numpy (so the numbers differ from gen.py's, the
distributions do not):
  * cluster centroids: unit-norm Gaussian directions, per head;
  * frame 0 keys: centroid of a uniformly drawn cluster + N(0, sigma^2 I);
  * frame f keys: a random permutation of frame f-1's stored keys plus
    N(0, frame_noise^2 I); a fraction `redraw` of the positions (drawn
    without replacement) is replaced by fresh keys of fresh clusters;
  * values N(0, 1); query i of frame f: centroid of key i's cluster +
    N(0, sigma^2 I); prompt keys from the same mixture, prompt values N(0, 1);
  * hyperplanes N(0, 1), one set [T*B][D] per layer.
Every array is rounded once to the storage type (bf16 round-to-nearest-even
by torch's conversion).  Like gen.py this module holds none of the method's
arithmetic.  Heads are drawn together (one [H][n][D] draw per frame), so a
layer's data does not depend on how its heads are later split over GPUs.
"""
from __future__ import annotations

import numpy as np
import torch

from .gen import ROOT_SEED, Config


def _seed(cfg: Config, layer: int, purpose: int) -> int:
    ss = np.random.SeedSequence([ROOT_SEED, cfg.idx, layer, 0xD0, purpose])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & 0x7FFFFFFFFFFFFFFF)


class DeviceLayerStream:
    """Frames of every head of one layer, drawn on `device` in order 0, 1, ..."""

    def __init__(self, cfg: Config, layer: int, device="cuda"):
        self.cfg, self.layer, self.device = cfg, layer, torch.device(device)
        self.dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        self.g = torch.Generator(device=self.device)
        self.g.manual_seed(_seed(cfg, layer, 1))
        c = self._randn(cfg.H, cfg.clusters, cfg.D)
        self.centroids = c / c.norm(dim=-1, keepdim=True)
        self._keys = None   # stored keys of the last frame (float32 holding storage values)
        self._clus = None

    def _randn(self, *shape):
        return torch.randn(*shape, generator=self.g, device=self.device, dtype=torch.float32)

    def _gather_centroids(self, clus):
        H, n = clus.shape
        return torch.gather(self.centroids, 1, clus[..., None].expand(H, n, self.cfg.D))

    def _fresh(self, n):
        cfg = self.cfg
        clus = torch.randint(0, cfg.clusters, (cfg.H, n), generator=self.g, device=self.device)
        return clus, self._gather_centroids(clus) + cfg.sigma * self._randn(cfg.H, n, cfg.D)

    def frame(self):
        """(keys, values, queries) of the next frame, each [H][n_f][D] in the storage type."""
        cfg = self.cfg
        H, n, D = cfg.H, cfg.n_f, cfg.D
        if self._keys is None:
            clus, k = self._fresh(n)
        else:
            perm = torch.argsort(torch.rand(H, n, generator=self.g, device=self.device), dim=1)
            k = torch.gather(self._keys, 1, perm[..., None].expand(H, n, D))
            k = k + cfg.frame_noise * self._randn(H, n, D)
            clus = torch.gather(self._clus, 1, perm)
            nred = int(round(cfg.redraw * n))
            if nred:
                pos = torch.argsort(torch.rand(H, n, generator=self.g, device=self.device), dim=1)[:, :nred]
                c2, k2 = self._fresh(nred)
                k.scatter_(1, pos[..., None].expand(H, nred, D), k2)
                clus.scatter_(1, pos, c2)
        k = k.to(self.dt)
        v = self._randn(H, n, D).to(self.dt)
        q = (self._gather_centroids(clus) + cfg.sigma * self._randn(H, n, D)).to(self.dt)
        self._keys, self._clus = k.float(), clus
        return k, v, q

    def prompt(self):
        """Prompt keys and values [H][P][D] from the same mixture."""
        cfg = self.cfg
        g = torch.Generator(device=self.device)
        g.manual_seed(_seed(cfg, self.layer, 4))
        clus = torch.randint(0, cfg.clusters, (cfg.H, cfg.P), generator=g, device=self.device)
        k = self._gather_centroids(clus) + cfg.sigma * torch.randn(cfg.H, cfg.P, cfg.D, generator=g,
                                                                    device=self.device)
        v = torch.randn(cfg.H, cfg.P, cfg.D, generator=g, device=self.device)
        return k.to(self.dt), v.to(self.dt)

    def planes(self):
        g = torch.Generator(device=self.device)
        g.manual_seed(_seed(self.cfg, self.layer, 9))
        r = torch.randn(self.cfg.T * self.cfg.B, self.cfg.D, generator=g, device=self.device)
        return r.to(self.dt)
