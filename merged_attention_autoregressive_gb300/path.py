"""One chunk of the FAST-AR attention path on preallocated device buffers.

The order follows the method: hash the chunk's queries, its new keys and
the prompt keys once (FAST-AR analysis, paper.rainbus.top: the encoding is
computed once and serves all three modules); merge the new frames into the
TempCache; prune the prompt per frame (AnnCA); cross-attend; then
self-attend over the merged cache with the bucket restriction (AnnSA).
Every step is one C-ABI call; this class only owns the buffers.
"""
from __future__ import annotations

from types import SimpleNamespace

import torch

from . import (Cache, OP_ANNCA, OP_ANNSA, OP_ANNSA_PARTS, OP_MERGE, fastar_annca_attention, fastar_annca_prune,
               fastar_annsa_attention, fastar_annsa_attention_part, fastar_annsa_combine, fastar_bucket_csr,
               fastar_hash, fastar_hash_many, fastar_tempcache_merge, fastar_workspace_size)

DENSE_FRAC = 0.3  # sparse attention is off for this share of a chunk's denoising steps


class ChunkPath:
    """Buffers and calls of one layer's per-chunk path."""

    def __init__(self, H, D, n_f, F, P, T, B, C, tau, dtype=torch.bfloat16, device="cuda", rep="last",
                 share=None, search="prev"):
        """rep: TempCache representative, "last" (the method) or "mean";
        search: where a new key's group is looked for, "prev" (the previous
        frame's groups, the method) or "lsh" (every earlier group sharing an
        LSH bucket);
        share: another ChunkPath of the same shapes whose workspaces and
        streams this one reuses (layers run one after the other on the same
        streams, so their scratch never overlaps in time); caches, codes,
        outputs and events stay per layer."""
        self.H, self.D, self.n_f, self.F, self.P = H, D, n_f, F, P
        self.rep = rep  # TempCache representative: "last" (the method) or "mean" (ablation)
        self.search = search
        self.T, self.B, self.C, self.tau, self.dtype = T, B, C, tau, dtype
        self.Nq = F * n_f
        self.scale = D ** -0.5
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.cache = Cache(H, C, D, T, B, dtype, dev)
        self.planes = torch.zeros(T * B, D, dtype=dtype, device=dev)
        Nq = self.Nq
        self.q_codes = torch.zeros(H, T, Nq, **i32)
        self.q_perm = torch.zeros(H, T, Nq, **i32)
        self.q_offsets = torch.zeros(H, T, (1 << B) + 1, **i32)
        self.k_codes = torch.zeros(H, T, Nq, **i32)
        self.p_codes = torch.zeros(H, T, max(P, 1), **i32)
        self.kept_idx = torch.zeros(H, F, max(P, 1), **i32)
        self.kept_cnt = torch.zeros(H, F, **i32)
        self.match = torch.zeros(H, Nq, **i32)
        self.o_ca = torch.zeros(H, Nq, D, dtype=dtype, device=dev)
        self.o_sa = torch.zeros(H, Nq, D, dtype=dtype, device=dev)
        self.lse = torch.zeros(H, Nq, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, **i32)
        if share is not None:
            if (share.H, share.D, share.n_f, share.F, share.P, share.T, share.B, share.C) != \
                    (H, D, n_f, F, P, T, B, C):
                raise ValueError("a shared path must have the same shapes")
            self.ws_merge, self.ws_annsa, self.ws_annca = share.ws_merge, share.ws_annsa, share.ws_annca
            self._side, self._copy_in, self._copy_out = share._side, share._copy_in, share._copy_out
        else:
            self.ws_merge = torch.empty(max(1, fastar_workspace_size(OP_MERGE, H, n_f, D, T, B, C)),
                                        dtype=torch.uint8, device=dev)
            self.ws_annsa = torch.empty(max(1, fastar_workspace_size(OP_ANNSA, H, Nq, D, T, B, C)),
                                        dtype=torch.uint8, device=dev)
            self.ws_annca = torch.empty(max(1, fastar_workspace_size(OP_ANNCA, H, F, D, T, B, P)),
                                        dtype=torch.uint8, device=dev)
            # the second stream (query CSR, cross-attention branch)
            self._side = torch.cuda.Stream(device=dev)
            # host-to-host chunks: the streams that copy inputs in and outputs out
            self._copy_in = torch.cuda.Stream(device=dev)
            self._copy_out = torch.cuda.Stream(device=dev)
        # the events that fork and join the second stream
        self._fork = torch.cuda.Event()
        self._codes_ready = torch.cuda.Event()
        self._csr_done = torch.cuda.Event()
        # host-to-host chunks: device copies of the inputs and the events
        # that release each branch and each output
        self._dev_in = None
        self._in_k = torch.cuda.Event()
        self._in_v = torch.cuda.Event()
        self._in_qp = torch.cuda.Event()
        self._in_vp = torch.cuda.Event()
        self._cross_done = torch.cuda.Event()
        self._ca_done = torch.cuda.Event()
        self._sa_done = torch.cuda.Event()
        self._out_done = torch.cuda.Event()

    # -- pieces -----------------------------------------------------------
    def merge(self, k, v, first_frame, F=None, stream=None):
        """Hash new keys k [H][F*n_f][D] and merge them (cache building).

        Returns (codes [H][T][F*n_f], match [H][F*n_f]) of this call.
        """
        F = self.F if F is None else F
        n = F * self.n_f
        if F == self.F:
            codes, match = self.k_codes, self.match
        else:
            codes = torch.empty(self.H, self.T, n, dtype=torch.int32, device=k.device)
            match = torch.empty(self.H, n, dtype=torch.int32, device=k.device)
        fastar_hash(k, self.planes, self.T, self.B, codes, status=self.status, stream=stream)
        fastar_tempcache_merge(self.cache, k, v, codes, F, self.n_f, first_frame, self.tau,
                               match_out=match, ws=self.ws_merge, status=self.status,
                               stream=stream, rep=self.rep, planes=self.planes,
                               search=self.search)
        return codes, match

    def step(self, q, k, v, kp, vp, first_frame, stream=None):
        """The whole path for one chunk: q, k, v [H][F*n_f][D]; kp, vp [H][P][D].

        The second stream hashes the chunk while the merge starts (its first
        NN search and plan need only the keys and the cache; it waits for
        the key codes before its first apply), then builds the query CSR and
        runs the cross-attention branch (prune, AnnCA), which needs the codes
        but not the merged cache; AnnSA waits for the CSR, and `stream`
        (default: the current stream) waits for both branches before this
        returns, so later work on it sees every output."""
        self._run(q, k, v, kp, vp, first_frame, self._main(stream))

    def step_host(self, hq, hk, hv, hkp, hvp, ho_ca, ho_sa, first_frame, stream=None, dev_in=None,
                  join=True):
        """The chunk from host memory to host memory (pinned tensors, same
        shapes as step's; ho_ca, ho_sa receive o_ca and o_sa).

        The inputs are copied in on one copy stream in the order the
        branches need them (k and v for the merge branch, then q, the prompt
        keys and the prompt values for the cross-attention branch, which
        also builds the query CSR that AnnSA needs; one host-to-device stream
        beside the device-to-host one moves more in total than two), each
        branch hashes and starts as soon as its inputs have landed, and each
        output is copied out on a second stream as soon as it is final.  The copies into this
        path's device buffers (dev_in: (q, k, v, kp, vp) tensors to use; by
        default buffers of its own) wait only for the previous chunk of this
        path to have read them, so with several paths (layers) the copies of
        one run ahead of the kernels of another.  With join (the default)
        `stream` (default: the current stream) waits for all of it, so the
        host buffers are complete once it has synchronised; without, call
        join_outputs before reading them."""
        main = self._main(stream)
        dev = self.q_codes.device
        if dev_in is not None:
            self._dev_in = list(dev_in)
        elif self._dev_in is None or self._dev_in[0].shape != hq.shape or self._dev_in[3].shape != hkp.shape:
            self._dev_in = [torch.empty(x.shape, dtype=x.dtype, device=dev) for x in (hq, hk, hv, hkp, hvp)]
        dq, dk, dv, dkp, dvp = self._dev_in
        # the device inputs and outputs are free once this path's previous
        # chunk has finished and its outputs have been copied out (never
        # recorded before the first chunk); every stream of this chunk waits
        # for that through the copies it depends on
        ci = self._copy_in
        ci.wait_event(self._out_done)
        with torch.cuda.stream(ci):
            dk.copy_(hk, non_blocking=True)
            self._in_k.record(ci)
            dv.copy_(hv, non_blocking=True)
            self._in_v.record(ci)
            dq.copy_(hq, non_blocking=True)
            dkp.copy_(hkp, non_blocking=True)
            self._in_qp.record(ci)
            dvp.copy_(hvp, non_blocking=True)
            self._in_vp.record(ci)
        main.wait_event(self._out_done)
        self._run(dq, dk, dv, dkp, dvp, first_frame, main, host_out=(ho_ca, ho_sa))
        co = self._copy_out
        co.wait_event(self._ca_done)
        with torch.cuda.stream(co):
            ho_ca.copy_(self.o_ca, non_blocking=True)
        co.wait_event(self._sa_done)
        with torch.cuda.stream(co):
            ho_sa.copy_(self.o_sa, non_blocking=True)
        self._out_done.record(co)
        if join:
            self.join_outputs(main)

    def join_outputs(self, stream=None):
        """Make `stream` (default: the current stream) wait until the host
        outputs of this path's last step_host are complete."""
        self._main(stream).wait_event(self._out_done)

    # -- denoising steps -----------------------------------------------------
    def denoise_step(self, s, S, q, k, v, kp, vp, first_frame, dense_frac=DENSE_FRAC, reuse=False):
        """Step s of the S denoising steps of a chunk (FAST-AR analysis,
        paper.rainbus.top: sparse attention is off for the first 30 % of the
        steps; each chunk is denoised conditioned on the history).

        Step s is dense iff s < dense_frac * S.  A step before the last
        attends the cache together with its own keys (count 1; the cache is
        not written): two partial AnnSA calls, one over the cache and one
        over a cache description of the step's keys, merged exactly by
        fastar_annsa_combine; dense steps give both key sets one table of one
        bit with every code 0, and keep every prompt token.  The last step
        merges its keys into the cache and attends the merged cache, as
        `step` does (dense per the schedule).  Outputs: o_sa, lse, o_ca.

        reuse: the codes (queries, the step's keys, the prompt), the query
        CSR and the kept prompt lists are computed at the chunk's first
        sparse step only and reused by its later sparse steps; the last step
        still hashes its keys, whose codes the merge stores with them."""
        dense = s < dense_frac * S
        first_sparse = not dense and (s == 0 or (s - 1) < dense_frac * S)
        reuse_now = reuse and not dense and not first_sparse
        dn = self._denoise_views()
        st = self.status
        if s + 1 == S and not dense:
            if not reuse_now:
                self.step(q, k, v, kp, vp, first_frame)
                return
            fastar_hash(k, self.planes, self.T, self.B, self.k_codes, status=st)
            fastar_tempcache_merge(self.cache, k, v, self.k_codes, self.F, self.n_f, first_frame, self.tau,
                                   match_out=self.match, ws=self.ws_merge, status=st, rep=self.rep,
                                   planes=self.planes, search=self.search)
            fastar_annsa_attention(q, self.q_codes, self.q_perm, self.q_offsets, self.cache, self.scale, self.o_sa,
                                   self.lse, ws=self.ws_annsa, status=st)
            fastar_annca_attention(q, kp, vp, self.kept_idx, self.kept_cnt, self.F, self.n_f, self.scale,
                                   self.o_ca, ws=self.ws_annca, status=st)
            return
        if s + 1 == S:
            fastar_hash(k, self.planes, self.T, self.B, self.k_codes, status=st)
            fastar_tempcache_merge(self.cache, k, v, self.k_codes, self.F, self.n_f, first_frame, self.tau,
                                   match_out=self.match, ws=self.ws_merge, status=st, rep=self.rep,
                                   planes=self.planes)
            fastar_annsa_attention_part(q, dn.qc0, dn.qp0, dn.qo0, dn.cache_dense, self.scale, 0, 1, dn.ws,
                                        status=st)
            fastar_annsa_combine(1, dn.ws, self.o_sa, self.lse, status=st)
        elif dense:
            chunk = self._chunk_view(k, v, dense=True)
            fastar_annsa_attention_part(q, dn.qc0, dn.qp0, dn.qo0, dn.cache_dense, self.scale, 0, 2, dn.ws,
                                        status=st)
            fastar_annsa_attention_part(q, dn.qc0, dn.qp0, dn.qo0, chunk, self.scale, 1, 2, dn.ws, status=st)
            fastar_annsa_combine(2, dn.ws, self.o_sa, self.lse, status=st)
        else:
            T = self.T
            jobs = [(q, self.q_codes, self.q_perm, self.q_offsets), (k, self.k_codes, dn.k_perm, dn.k_off)]
            if self.P:
                jobs.append((kp, self.p_codes, None, None))
            if not reuse_now:
                fastar_hash_many(jobs, self.planes, T, self.B, status=st)
            chunk = self._chunk_view(k, v, dense=False)
            fastar_annsa_attention_part(q, self.q_codes, self.q_perm, self.q_offsets, self.cache, self.scale, 0,
                                        2 * T, dn.ws, status=st)
            fastar_annsa_attention_part(q, self.q_codes, self.q_perm, self.q_offsets, chunk, self.scale, T,
                                        2 * T, dn.ws, status=st)
            fastar_annsa_combine(2 * T, dn.ws, self.o_sa, self.lse, status=st)
        if dense:
            kept, cnt = dn.kept_all, dn.cnt_all
        elif reuse_now:
            kept, cnt = self.kept_idx, self.kept_cnt
        else:
            fastar_annca_prune(self.q_codes, self.p_codes[:, :, :self.P], self.F, self.n_f, self.B,
                               self.kept_idx, self.kept_cnt, status=st)
            kept, cnt = self.kept_idx, self.kept_cnt
        fastar_annca_attention(q, kp, vp, kept, cnt, self.F, self.n_f, self.scale, self.o_ca, ws=self.ws_annca,
                               status=st)

    def _chunk_view(self, k, v, dense):
        dn = self._denoise_views()
        if dense:
            return Cache.view(1, 1, K=k, V=v, m=dn.ones, codes=dn.qc0, last_frame=dn.lf, size=dn.nq,
                              inserted=dn.cnt64, evicted=dn.cnt64, perm=dn.qp0, offsets=dn.qo0)
        return Cache.view(self.T, self.B, K=k, V=v, m=dn.ones, codes=self.k_codes, last_frame=dn.lf,
                          size=dn.nq, inserted=dn.cnt64, evicted=dn.cnt64, perm=dn.k_perm, offsets=dn.k_off)

    def _denoise_views(self):
        """Buffers of the denoising steps, built once: one-bucket (dense)
        views of the queries, of the cache and of a step's keys (codes 0; the
        CSR kernel turns them into an identity order and offsets (0, N, N)),
        every prompt token kept (the prune of all-zero codes), and a step's
        keys described as a cache (m = 1, size = Nq, their own CSR)."""
        if getattr(self, "_dn", None) is not None:
            return self._dn
        if 2 * self.T > 4:
            raise ValueError("denoising steps need T <= 2 (2 T partial results per query)")
        H, C, Nq, F, P, D = self.H, self.C, self.Nq, self.F, self.P, self.D
        dev = self.q_codes.device
        i32 = dict(dtype=torch.int32, device=dev)
        dn = SimpleNamespace()

        def one_bucket(n):
            codes = torch.zeros(H, 1, n, **i32)
            perm = torch.empty(H, 1, n, **i32)
            off = torch.empty(H, 1, 3, **i32)
            fastar_bucket_csr(codes, 1, perm, off, status=self.status)
            return codes, perm, off

        dn.qc0, dn.qp0, dn.qo0 = one_bucket(Nq)
        cc0, cp0, co0 = one_bucket(C)
        c = self.cache
        dn.cache_dense = Cache.view(1, 1, K=c.K, V=c.V, m=c.m, codes=cc0, last_frame=c.last_frame, size=c.size,
                                    inserted=c.inserted, evicted=c.evicted, perm=cp0, offsets=co0)
        dn.kept_all = torch.empty(H, F, max(P, 1), **i32)
        dn.cnt_all = torch.empty(H, F, **i32)
        fastar_annca_prune(dn.qc0, torch.zeros(H, 1, P, **i32), F, self.n_f, 1, dn.kept_all, dn.cnt_all,
                           status=self.status)
        dn.ones = torch.ones(H, Nq, **i32)
        dn.lf = torch.zeros(H, Nq, **i32)
        dn.nq = torch.full((H,), Nq, **i32)
        dn.cnt64 = torch.zeros(H, dtype=torch.int64, device=dev)
        dn.k_perm = torch.empty(H, self.T, Nq, **i32)
        dn.k_off = torch.empty(H, self.T, (1 << self.B) + 1, **i32)
        dn.ws = torch.empty(fastar_workspace_size(OP_ANNSA_PARTS, H, Nq, D, 2 * self.T, self.B, C),
                            dtype=torch.uint8, device=dev)
        self._dn = dn
        return dn

    # -- internals ----------------------------------------------------------
    @staticmethod
    def _main(stream):
        if stream is None:
            return torch.cuda.current_stream()
        return stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(int(stream))

    def _run(self, q, k, v, kp, vp, first_frame, main, host_out=None):
        st = self.status
        staged = host_out is not None
        side = self._side
        cross = [(q, self.q_codes, None, None)]
        if self.P:
            cross.append((kp, self.p_codes, None, None))
        # The second stream hashes the chunk while the merge starts on `main`
        # (candidate setup, the first frame's NN search and plan need only k
        # and the cache); the merge waits for the key codes (and v) right
        # before its first apply.
        # the second stream starts after the work already on `main` (so that
        # layers run one after the other, as in a model)
        self._fork.record(main)
        side.wait_event(self._fork)
        if staged:
            main.wait_event(self._in_k)
            side.wait_event(self._in_k)
            fastar_hash_many([(k, self.k_codes, None, None)], self.planes, self.T, self.B, status=st,
                             stream=side)
            side.wait_event(self._in_v)
            self._codes_ready.record(side)
            side.wait_event(self._in_qp)
            fastar_hash_many(cross, self.planes, self.T, self.B, status=st, stream=side)
        else:
            fastar_hash_many([(k, self.k_codes, None, None)] + cross, self.planes, self.T, self.B,
                             status=st, stream=side)
            self._codes_ready.record(side)
        fastar_bucket_csr(self.q_codes, self.B, self.q_perm, self.q_offsets, status=st, stream=side)
        self._csr_done.record(side)
        fastar_annca_prune(self.q_codes, self.p_codes[:, :, :self.P], self.F, self.n_f, self.B,
                           self.kept_idx, self.kept_cnt, status=st, stream=side)
        if staged:
            side.wait_event(self._in_vp)
        fastar_annca_attention(q, kp, vp, self.kept_idx, self.kept_cnt, self.F, self.n_f,
                               self.scale, self.o_ca, ws=self.ws_annca, status=st, stream=side)
        if staged:
            self._ca_done.record(side)
        self._cross_done.record(side)
        fastar_tempcache_merge(self.cache, k, v, self.k_codes, self.F, self.n_f, first_frame,
                               self.tau, match_out=self.match, ws=self.ws_merge, status=st,
                               stream=main, codes_ready=self._codes_ready, rep=self.rep, planes=self.planes,
                               search=self.search)
        main.wait_event(self._csr_done)
        fastar_annsa_attention(q, self.q_codes, self.q_perm, self.q_offsets, self.cache,
                               self.scale, self.o_sa, self.lse, ws=self.ws_annsa, status=st,
                               stream=main)
        if staged:
            self._sa_done.record(main)
        main.wait_event(self._cross_done)


class ChunkStack:
    """The per-chunk path of several independent layers of one model.

    One ChunkPath per layer (own cache, codes and outputs) sharing one set
    of workspaces and streams; `step` runs the layers one after the other on
    the calling stream, as the attention layers of a model run (a layer's
    second stream starts after the previous layer's work)."""

    def __init__(self, layers, H, D, n_f, F, P, T, B, C, tau, dtype=torch.bfloat16, device="cuda", rep="last",
                 search="prev"):
        self.paths = []
        for _ in range(layers):
            self.paths.append(ChunkPath(H, D, n_f, F, P, T, B, C, tau, dtype, device, rep,
                                        share=self.paths[0] if self.paths else None, search=search))

    def __len__(self):
        return len(self.paths)

    def step(self, inputs, first_frame, stream=None):
        """inputs[l] = (q, k, v, kp, vp) of layer l, as for ChunkPath.step."""
        if len(inputs) != len(self.paths):
            raise ValueError("one input tuple per layer")
        for p, x in zip(self.paths, inputs):
            p.step(*x, first_frame, stream=stream)

    def step_host(self, host_inputs, host_outputs, first_frame, stream=None, dev_in=None):
        """Host-to-host chunk of every layer: host_inputs[l] = (q, k, v, kp,
        vp) pinned, host_outputs[l] = (o_ca, o_sa) pinned; dev_in[l] optional
        device buffers for layer l's inputs.  The copies of later layers run
        ahead of the kernels of earlier ones; `stream` waits for every output."""
        if len(host_inputs) != len(self.paths) or len(host_outputs) != len(self.paths):
            raise ValueError("one input and one output tuple per layer")
        for i, p in enumerate(self.paths):
            p.step_host(*host_inputs[i], *host_outputs[i], first_frame, stream=stream,
                        dev_in=None if dev_in is None else dev_in[i], join=False)
        for p in self.paths:
            p.join_outputs(stream)
