"""fp64 CPU oracle of the FAST-AR per-chunk attention path.

TEST INFRASTRUCTURE ONLY.  Only the tests, `__graft_entry__.smoke()` and the
CPU-baseline leg of `bench.py` may import this module.  The CUDA library
never calls it and shares no code with it.

Every function is the plain definition of one step, written with numpy in
float64 (library matmul/sort/isin serve as steps; nothing is blocked, fused
or reordered beyond the definition).  Inputs are the exact stored values
(bf16 or fp32) widened to float64.

Sources (page title, then section):
  [PL]  FAST-AR summary on paperlayer.ai (arXiv 2602.01801v2)
  [GS]  FAST-AR "Technische samenvatting" on gist.science
  [RB]  FAST-AR analysis on paper.rainbus.top, "method steps" (方法步骤详情)

Readings taken where the pages are silent:
  hash    -- bit b of table t is [R_{t*B+b} . x > 0] (a zero dot gives 0),
             least significant bit = hyperplane t*B+0; one hyperplane set is
             shared by queries, cached keys and prompt keys.
  NN      -- new-frame *keys* are matched (cosine) against the
             representatives refreshed in frame f-1; ties go to the lowest
             slot; matched iff cosine >= tau; no merging inside a frame.
  merge   -- all keys matching one group join it; the representative key
             becomes the matching key with the lowest token index; the
             stored value is the count-weighted mean rounded to the storage
             type after each update.
  mean-key -- the representative ablation ([PL] appendix C, representative
             selection: last-key, mean-key, medoid-key): in "mean" mode the
             stored key is the count-weighted mean of every key that joined
             the group, updated and rounded like the value, and the group's
             codes are the hash of that stored key (its bucket).  The
             medoid-key variant needs every past member and is not built.
  denoise  -- step s of S is dense iff s < 0.3 S; a step before the last
             attends the cache plus its own keys and writes nothing; the
             last step merges and attends the merged cache.
  quant    -- the quantised matcher: per-dimension uniform b-bit codes over
             the searched vectors' own range; approximate scores on the
             decoded vectors; top-k per query (ties: lower index), attended
             exactly; TempCache takes the approximate top-1 and merges iff
             its exact cosine reaches tau.
  insert  -- unmatched keys fill free slots in ascending order, then the
             slots with the smallest (last_frame, slot) among those not
             refreshed in this frame are evicted (least recently refreshed).
  attend  -- a chunk's frames are merged first, then its queries attend the
             whole live cache; logit = q.k / sqrt(D) + ln m; a query with no
             allowed key gets a zero output and lse = -inf.
  recall  -- the pages report recall and density of the sparse selections
             without a formula; here a query's retained share is the dense
             softmax weight (same logits) on its allowed keys, and density is
             the allowed share of the (query, key) pairs.

Parity pins of every function live in tests/test_oracle_pins.py; there is
no worked numeric example on the pages, so the pins are closed forms
(Lemma 5.1), brute force on tiny inputs, invariants and hand-derived
fixtures under tests/golden/.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

HASH_MARGIN = 1e-4   # relative |R.x| / (|R| |x|) below which a bit is listed
NN_MARGIN = 1e-4     # cosine gap below which an NN decision is listed


# --------------------------------------------------------------------------
# storage rounding (the cache stores merged values in the input type)
# --------------------------------------------------------------------------
def round_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to bf16 or fp32, round-to-nearest-even ("f64": as is).

    bf16 keeps 8 significant bits: write x = mant * 2**e with mant in
    [0.5, 1), round mant * 2**8 to the nearest integer (ties to even) and
    scale back.  Exact for every finite value this path produces.
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f64":          # unrounded storage (closed-form checks only)
        return x
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype != "bf16":
        raise ValueError(dtype)
    mant, e = np.frexp(x)
    return np.ldexp(np.rint(mant * 256.0), e - 8)


# --------------------------------------------------------------------------
# step 1: random-hyperplane LSH  ([PL] section 2 "ANN search", section 5
# "ANN Attention"; [GS] 2.B mechanism: queries and prompt keys projected
# into one shared LSH space; [RB] technical novelty: the encoding is
# computed once and used by all three modules)
# --------------------------------------------------------------------------
def hash_codes(x: np.ndarray, planes: np.ndarray, T: int, B: int):
    """codes[h][t][i] = sum_b [planes[t*B+b] . x[h][i] > 0] << b.

    x: [H][N][D], planes: [T*B][D].  Returns (codes uint32 [H][T][N],
    margin_bits uint32 [H][T][N]) where a margin bit marks a dot product
    with |s| < HASH_MARGIN * |R| * |x| (either bit value is accepted there).
    """
    x = np.asarray(x, dtype=np.float64)
    R = np.asarray(planes, dtype=np.float64)
    H, N, D = x.shape
    assert R.shape == (T * B, D)
    s = np.einsum("hnd,rd->hrn", x, R)                      # [H][T*B][N]
    bits = (s > 0).astype(np.uint64)
    thr = HASH_MARGIN * np.linalg.norm(R, axis=1)[None, :, None] \
        * np.linalg.norm(x, axis=2)[:, None, :]
    near = (np.abs(s) < thr).astype(np.uint64)
    codes = np.zeros((H, T, N), dtype=np.uint64)
    margin = np.zeros((H, T, N), dtype=np.uint64)
    for t in range(T):
        for b in range(B):
            codes[:, t, :] |= bits[:, t * B + b, :] << np.uint64(b)
            margin[:, t, :] |= near[:, t * B + b, :] << np.uint64(b)
    return codes.astype(np.uint32), margin.astype(np.uint32)


# --------------------------------------------------------------------------
# step 2: bucket CSR (ids grouped by code, stable)
# --------------------------------------------------------------------------
def bucket_csr(codes: np.ndarray, nbuckets: int, n: int | None = None):
    """Stable grouping of ids 0..n-1 by code.

    codes: [..., N].  Returns perm [..., N] (entries past n are -1) and
    offsets [..., nbuckets+1] with offsets[c] = #ids (< n) whose code < c.
    """
    codes = np.asarray(codes)
    lead = codes.shape[:-1]
    N = codes.shape[-1]
    n = N if n is None else n
    flat = codes.reshape(-1, N)
    perm = np.full(flat.shape, -1, dtype=np.int32)
    offs = np.zeros((flat.shape[0], nbuckets + 1), dtype=np.int32)
    for g in range(flat.shape[0]):
        c = flat[g, :n].astype(np.int64)
        perm[g, :n] = np.argsort(c, kind="stable")
        offs[g, 1:] = np.cumsum(np.bincount(c, minlength=nbuckets)[:nbuckets])
    return perm.reshape(lead + (N,)), offs.reshape(lead + (nbuckets + 1,))


# --------------------------------------------------------------------------
# TempCache state ([PL] section 5 "TempCache" and appendix A, Lemma 5.1;
# [GS] 2.A; [RB] method steps, TempCache)
# --------------------------------------------------------------------------
@dataclass
class CacheState:
    """Fixed-capacity merged cache of one layer (all heads).

    K, V: [H][C][D] float64 holding stored (bf16/fp32) values.
    m: [H][C] group counts; codes: [H][T][C]; last_frame: [H][C] (-1 empty);
    size: [H] live slots (slots >= size are empty); inserted/evicted: [H].
    """
    dtype: str
    K: np.ndarray
    V: np.ndarray
    m: np.ndarray
    codes: np.ndarray
    last_frame: np.ndarray
    size: np.ndarray
    inserted: np.ndarray
    evicted: np.ndarray

    @staticmethod
    def empty(H: int, C: int, D: int, T: int, dtype: str) -> "CacheState":
        return CacheState(dtype, np.zeros((H, C, D)), np.zeros((H, C, D)),
                          np.zeros((H, C), np.int64), np.zeros((H, T, C), np.uint32),
                          np.full((H, C), -1, np.int64), np.zeros(H, np.int64),
                          np.zeros(H, np.int64), np.zeros(H, np.int64))

    def copy(self) -> "CacheState":
        return dataclasses.replace(self, **{f.name: np.copy(getattr(self, f.name))
                                            for f in dataclasses.fields(self)
                                            if f.name != "dtype"})

    @property
    def H(self):
        return self.K.shape[0]

    @property
    def C(self):
        return self.K.shape[1]


class CapacityError(RuntimeError):
    pass


def tempcache_nn(state: CacheState, k: np.ndarray, f: int, tau: float):
    """Top-1 cosine match of frame f's keys against frame f-1's representatives.

    k: [H][n][D].  Candidates of head h are the live slots s (s < size)
    with last_frame[s] == f-1, in ascending s.  Returns (match [H][n] slot
    or -1, listed [H][n] bool).  A decision is listed when the top-1 cosine
    is within NN_MARGIN of tau, or when the top-2 gap is below NN_MARGIN and
    the top-1 cosine is at least tau - NN_MARGIN.
    """
    k = np.asarray(k, dtype=np.float64)
    H, n, D = k.shape
    match = np.full((H, n), -1, dtype=np.int64)
    listed = np.zeros((H, n), dtype=bool)
    for h in range(H):
        size = int(state.size[h])
        cand = np.nonzero(state.last_frame[h, :size] == f - 1)[0]
        if cand.size == 0:
            continue
        Kc = state.K[h, cand]
        kn = np.linalg.norm(k[h], axis=1)
        cn = np.linalg.norm(Kc, axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            cos = (k[h] @ Kc.T) / (kn[:, None] * cn[None, :])
        cos[~np.isfinite(cos)] = -np.inf          # zero norm: no similarity
        best = np.argmax(cos, axis=1)              # first max = lowest slot
        top1 = cos[np.arange(n), best]
        ok = top1 >= tau
        match[h, ok] = cand[best[ok]]
        near_tau = np.abs(top1 - tau) < NN_MARGIN
        if cand.size > 1:
            top2 = np.partition(cos, cand.size - 2, axis=1)    # [..., second, first]
            near_tie = (top2[:, -1] - top2[:, -2]) < NN_MARGIN
        else:
            near_tie = np.zeros(n, dtype=bool)
        # a near tie only matters when the best cosine can reach tau
        listed[h] = np.isfinite(top1) & (near_tau | (near_tie & (top1 >= tau - NN_MARGIN)))
    return match, listed


def tempcache_nn_lsh(state: CacheState, k: np.ndarray, k_codes: np.ndarray, f: int, tau: float):
    """The search variant that matches against every previous frame ([GS]
    2.A looks for the nearest key over the earlier frames with LSH or
    quantisation; the method's default takes only the previous frame, [RB]
    method steps): the candidates of key
    j are the live groups refreshed before frame f that share an LSH bucket
    with it in some table; top-1 cosine among them (ties: lowest slot),
    merged iff the cosine reaches tau.  k_codes: [H][T][n].  Returns
    (match [H][n], listed [H][n]) with the listing rule of tempcache_nn."""
    k = np.asarray(k, dtype=np.float64)
    H, n, D = k.shape
    match = np.full((H, n), -1, dtype=np.int64)
    listed = np.zeros((H, n), dtype=bool)
    for h in range(H):
        size = int(state.size[h])
        live = np.nonzero((state.last_frame[h, :size] >= 0) & (state.last_frame[h, :size] < f))[0]
        if live.size == 0:
            continue
        share = annsa_allowed(np.asarray(k_codes)[h], state.codes[h][:, live])   # [n][live]
        Kc = state.K[h, live]
        kn = np.linalg.norm(k[h], axis=1)
        cn = np.linalg.norm(Kc, axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            cos = (k[h] @ Kc.T) / (kn[:, None] * cn[None, :])
        cos[~np.isfinite(cos) | ~share] = -np.inf
        best = np.argmax(cos, axis=1)
        top1 = cos[np.arange(n), best]
        ok = top1 >= tau
        match[h, ok] = live[best[ok]]
        near_tau = np.abs(top1 - tau) < NN_MARGIN
        with np.errstate(invalid="ignore"):   # rows with fewer than two candidates: no tie
            if live.size > 1:
                top2 = np.partition(cos, live.size - 2, axis=1)    # [..., second, first]
                near_tie = (top2[:, -1] - top2[:, -2]) < NN_MARGIN
            else:
                near_tie = np.zeros(n, dtype=bool)
        listed[h] = np.isfinite(top1) & (near_tau | (near_tie & (top1 >= tau - NN_MARGIN)))
    return match, listed


def tempcache_apply_frame(state: CacheState, k, v, codes, f: int, match, rep: str = "last",
                          planes=None, B: int | None = None) -> CacheState:
    """Merge one frame's keys into the cache given its NN matches (in place).

    k, v: [H][n][D]; codes: [H][T][n]; match: [H][n] slot or -1.
    Matched groups (Lemma 5.1): m' = m + |S|, V' = round((m V + sum v)/m'),
    the representative key, its codes and last_frame come from the lowest
    matching index.  Unmatched keys become groups of count 1, placed in free
    slots first, then in evicted slots (smallest (last_frame, slot) among
    slots with last_frame < f), both in ascending order.
    rep="mean" ([PL] appendix C, mean-key representative): the matched
    group's key is K' = round((m K + sum k)/m') instead, and its codes are
    hash(K') with `planes` [T*B][D] and B bits per table.
    """
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    H, n, D = k.shape
    C = state.C
    for h in range(H):
        mh = np.asarray(match[h])
        for s in np.unique(mh[mh >= 0]):
            S = np.nonzero(mh == s)[0]              # ascending token index
            m_old = int(state.m[h, s])
            m_new = m_old + S.size
            total = m_old * state.V[h, s]
            for j in S:
                total = total + v[h, j]
            state.V[h, s] = round_storage(total / m_new, state.dtype)
            if rep == "mean":
                ktot = m_old * state.K[h, s]
                for j in S:
                    ktot = ktot + k[h, j]
                state.K[h, s] = round_storage(ktot / m_new, state.dtype)
                T = state.codes.shape[1]
                state.codes[h, :, s] = hash_codes(state.K[h, s][None, None], planes, T, B)[0][0, :, 0]
            else:
                state.K[h, s] = k[h, S[0]]
                state.codes[h, :, s] = codes[h, :, S[0]]
            state.last_frame[h, s] = f
            state.m[h, s] = m_new
        U = np.nonzero(mh < 0)[0]
        size = int(state.size[h])
        free = C - size
        n_app = min(free, U.size)
        targets = list(range(size, size + n_app))
        n_evict = U.size - n_app
        if n_evict > 0:
            lf = state.last_frame[h, :size]
            elig = np.nonzero(lf < f)[0]
            if elig.size < n_evict:
                raise CapacityError(f"head {h}: {n_evict} evictions needed, "
                                    f"{elig.size} slots evictable")
            order = np.lexsort((elig, lf[elig]))    # by last_frame, then slot
            targets += sorted(elig[order[:n_evict]].tolist())
        for r, j in enumerate(U):
            s = targets[r]
            if s < size:
                state.evicted[h] += state.m[h, s]
            state.K[h, s] = k[h, j]
            state.V[h, s] = v[h, j]
            state.m[h, s] = 1
            state.codes[h, :, s] = codes[h, :, j]
            state.last_frame[h, s] = f
        state.size[h] = size + n_app
        state.inserted[h] += n
    return state


def tempcache_merge(state: CacheState, k_new, v_new, codes_new, F: int, n_f: int,
                    first_frame: int, tau: float, match_override=None, rep: str = "last",
                    planes=None, B: int | None = None, search: str = "prev"):
    """Merge a chunk of F frames, frame by frame, into a copy of `state`.

    k_new, v_new: [H][F*n_f][D]; codes_new: [H][T][F*n_f].
    match_override: optional [H][F*n_f] matches to use instead of the
    oracle's own (to continue from another implementation's decisions).
    rep, planes, B: the representative mode (tempcache_apply_frame).
    search: "prev" (the method: frame f-1's groups, tempcache_nn), "lsh"
    (every earlier group sharing a bucket, tempcache_nn_lsh) or "quant<b>"
    (frame f-1's groups ranked by their b-bit codes, tempcache_nn_quant).
    Returns (new_state, match [H][F*n_f], listed [H][F*n_f]).
    """
    st = state.copy()
    H = st.H
    match = np.full((H, F * n_f), -1, dtype=np.int64)
    listed = np.zeros((H, F * n_f), dtype=bool)
    for fi in range(F):
        sl = slice(fi * n_f, (fi + 1) * n_f)
        f = first_frame + fi
        if search == "lsh":
            mt, ls = tempcache_nn_lsh(st, np.asarray(k_new)[:, sl], np.asarray(codes_new)[:, :, sl], f, tau)
        elif search.startswith("quant"):
            mt, ls = tempcache_nn_quant_listed(st, np.asarray(k_new)[:, sl], f, tau, int(search[5:]))
        elif search == "prev":
            mt, ls = tempcache_nn(st, np.asarray(k_new)[:, sl], f, tau)
        else:
            raise ValueError(search)
        if match_override is not None:
            mt = np.asarray(match_override)[:, sl].astype(np.int64)
        match[:, sl], listed[:, sl] = mt, ls
        tempcache_apply_frame(st, np.asarray(k_new)[:, sl], np.asarray(v_new)[:, sl],
                              np.asarray(codes_new)[:, :, sl], f, mt, rep=rep, planes=planes, B=B)
    return st, match, listed


# --------------------------------------------------------------------------
# step 5: AnnCA pruning ([GS] 2.B mechanism; [RB] method steps, AnnCA;
# [PL] section 5 "AnnCA")
# --------------------------------------------------------------------------
def annca_prune(q_codes, p_codes, F: int, n_f: int):
    """Per (head, frame): ascending prompt ids sharing >= 1 bucket with a query.

    q_codes: [H][T][F*n_f]; p_codes: [H][T][P].  A prompt token is kept
    for frame f iff for some table t its code equals the table-t code of
    at least one query of frame f.  Returns (kept_idx [H][F][P] padded
    with -1, kept_cnt [H][F]).
    """
    q_codes = np.asarray(q_codes)
    p_codes = np.asarray(p_codes)
    H, T, _ = q_codes.shape
    P = p_codes.shape[2]
    kept_idx = np.full((H, F, P), -1, dtype=np.int32)
    kept_cnt = np.zeros((H, F), dtype=np.int32)
    for h in range(H):
        for f in range(F):
            keep = np.zeros(P, dtype=bool)
            for t in range(T):
                occ = np.unique(q_codes[h, t, f * n_f:(f + 1) * n_f])
                keep |= np.isin(p_codes[h, t], occ)
            ids = np.nonzero(keep)[0]
            kept_idx[h, f, :ids.size] = ids
            kept_cnt[h, f] = ids.size
    return kept_idx, kept_cnt


# --------------------------------------------------------------------------
# steps 6-7: attention with an explicit allowed set and a logit bias
# ([PL] section 3 attention formulation; appendix A, Lemma A.1)
# --------------------------------------------------------------------------
def masked_attention(q, k, v, allowed, bias, scale: float):
    """o_i = sum_j softmax_j(scale q_i.k_j + bias_j | allowed_ij) v_j, in fp64.

    q: [n][D], k, v: [M][D], allowed: [n][M] bool, bias: [M].
    Rows with no allowed key give o = 0 and lse = -inf.
    Returns (o [n][D], lse [n]) with lse = ln sum_j exp(logit_j).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, D = q.shape
    if k.shape[0] == 0:
        return np.zeros((n, v.shape[1] if v.ndim == 2 else D)), np.full(n, -np.inf)
    s = scale * (q @ k.T) + np.asarray(bias, dtype=np.float64)[None, :]
    s = np.where(allowed, s, -np.inf)
    M = np.max(s, axis=1)
    anyk = np.isfinite(M)
    Ms = np.where(anyk, M, 0.0)
    w = np.where(allowed, np.exp(s - Ms[:, None]), 0.0)
    lsum = np.sum(w, axis=1)
    o = np.zeros((n, v.shape[1]))
    o[anyk] = (w[anyk] @ v) / lsum[anyk, None]
    lse = np.full(n, -np.inf)
    lse[anyk] = Ms[anyk] + np.log(lsum[anyk])
    return o, lse


def annca_attention(q, k_p, v_p, kept_idx, kept_cnt, F: int, n_f: int, scale: float,
                    rows=None):
    """Cross-attention of frame f's queries over its kept prompt tokens.

    q: [H][F*n_f][D]; k_p, v_p: [H][P][D]; kept_idx [H][F][P]; kept_cnt [H][F].
    `rows` optionally restricts the output to these query indices (same for
    every head).  Returns o [H][n][D] (n = F*n_f or len(rows)).
    """
    q = np.asarray(q, dtype=np.float64)
    H, Nq, D = q.shape
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    o = np.zeros((H, rows.size, np.asarray(v_p).shape[2]))
    for h in range(H):
        for f in range(F):
            sel = np.nonzero((rows >= f * n_f) & (rows < (f + 1) * n_f))[0]
            if sel.size == 0:
                continue
            ids = np.asarray(kept_idx[h, f, :kept_cnt[h, f]], dtype=np.int64)
            allowed = np.ones((sel.size, ids.size), dtype=bool)
            o[h, sel], _ = masked_attention(q[h, rows[sel]], np.asarray(k_p)[h, ids],
                                            np.asarray(v_p)[h, ids], allowed,
                                            np.zeros(ids.size), scale)
    return o


def annsa_allowed(q_codes_h, cache_codes_h):
    """allowed[i][s] = exists t: q_codes[t][i] == codes[t][s] (token-exact)."""
    T = q_codes_h.shape[0]
    allowed = np.zeros((q_codes_h.shape[1], cache_codes_h.shape[1]), dtype=bool)
    for t in range(T):
        allowed |= q_codes_h[t][:, None] == cache_codes_h[t][None, :]
    return allowed


def annsa_attention(q, q_codes, state: CacheState, scale: float, rows=None):
    """Bucket-restricted self-attention of the chunk's queries over the cache.

    A query may attend a live slot iff they share a code in some table
    ([GS] 2.C; [RB] method steps, AnnSA); logit = scale q.K[s] + ln m[s]
    (Lemma 5.1).  q: [H][Nq][D]; q_codes: [H][T][Nq].  `rows` optionally
    restricts the computation to a subset of query indices (same for all
    heads).  Returns (o [H][n][D], lse [H][n]).
    """
    q = np.asarray(q, dtype=np.float64)
    H, Nq, D = q.shape
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    o = np.zeros((H, rows.size, D))
    lse = np.zeros((H, rows.size))
    for h in range(H):
        size = int(state.size[h])
        allowed = annsa_allowed(np.asarray(q_codes)[h][:, rows], state.codes[h, :, :size])
        bias = np.log(state.m[h, :size].astype(np.float64))
        o[h], lse[h] = masked_attention(q[h, rows], state.K[h, :size], state.V[h, :size],
                                        allowed, bias, scale)
    return o, lse


# ---------------------------------------------------------------- denoising steps
# One chunk is denoised over S steps, each with its own queries, keys and
# values; generation is conditioned on the history in the cache ([PL]
# related work: chunked autoregressive denoising conditioned on previously
# generated history).  Sparse attention is off for the first 30 % of the
# denoising steps ([RB] limitations, fifth point).  Readings: step s is dense
# iff s < 0.3 S; a step before the last attends the cache's groups (+ ln m)
# together with its own keys (count 1) and writes nothing to the cache;
# the last step merges its keys into the cache (TempCache) and attends the
# merged cache, as the single-step chunk does.  A sparse step restricts
# self-attention to pairs that share a bucket in some table (on the cache
# and on its own keys alike) and cross-attention to each frame's kept prompt
# tokens; a dense step allows every live pair and every prompt token.
DENSE_FRAC = 0.3


def denoise_schedule(S: int, dense_frac: float = DENSE_FRAC):
    """dense[s] for the S denoising steps of a chunk: s < dense_frac * S."""
    return [s < dense_frac * S for s in range(S)]


def denoise_step_attention(q, q_codes, state: CacheState, k, v, k_codes, dense: bool, scale: float):
    """Self-attention of a non-final denoising step over the cache and the
    step's own keys (not merged).  q, k, v: [H][Nq][D]; q_codes, k_codes:
    [H][T][Nq].  Returns (o [H][Nq][D], lse [H][Nq])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    H, Nq, D = q.shape
    o = np.zeros((H, Nq, D))
    lse = np.zeros((H, Nq))
    for h in range(H):
        size = int(state.size[h])
        K = np.concatenate([state.K[h, :size], k[h]])
        V = np.concatenate([state.V[h, :size], v[h]])
        bias = np.concatenate([np.log(state.m[h, :size].astype(np.float64)), np.zeros(k.shape[1])])
        if dense:
            allowed = np.ones((Nq, K.shape[0]), dtype=bool)
        else:
            allowed = np.concatenate([annsa_allowed(np.asarray(q_codes)[h], state.codes[h, :, :size]),
                                      annsa_allowed(np.asarray(q_codes)[h], np.asarray(k_codes)[h])], axis=1)
        o[h], lse[h] = masked_attention(q[h], K, V, allowed, bias, scale)
    return o, lse


def denoise_chunk(state: CacheState, steps, k_p, v_p, planes, T: int, B: int, F: int, n_f: int,
                  first_frame: int, tau: float, scale: float, dense_frac: float = DENSE_FRAC,
                  reuse: bool = False):
    """The S denoising steps of one chunk.  steps: list of (q, k, v), each
    [H][F*n_f][D].  Returns (outs, final_state, match) where outs[s] =
    (o_sa, lse_sa, o_ca) and match is the final merge's.
    reuse: the codes of the queries and of the step's keys and the kept
    prompt lists of the chunk's first sparse step serve its later sparse
    steps too (the codes are computed once per chunk); the last step's keys
    are still hashed for the merge, which stores their codes."""
    dense = denoise_schedule(len(steps), dense_frac)
    pc, _ = hash_codes(k_p, planes, T, B)
    H, P = np.asarray(k_p).shape[:2]
    st = state
    outs = []
    match = None
    kept = None   # (qc, kc, idx, cnt) of the first sparse step, with reuse
    for s, (q, k, v) in enumerate(steps):
        if reuse and not dense[s] and kept is not None:
            qc, kc, idx, cnt = kept
            if s + 1 == len(steps):
                kc, _ = hash_codes(k, planes, T, B)
        else:
            qc, _ = hash_codes(q, planes, T, B)
            kc, _ = hash_codes(k, planes, T, B)
            if dense[s]:
                idx = np.tile(np.arange(P), (H, F, 1))
                cnt = np.full((H, F), P)
            else:
                idx, cnt = annca_prune(qc, pc, F, n_f)
                if reuse:
                    kept = (qc, kc, idx, cnt)
        o_ca = annca_attention(q, k_p, v_p, idx, cnt, F, n_f, scale)
        if s + 1 < len(steps):
            o_sa, lse = denoise_step_attention(q, qc, st, k, v, kc, dense[s], scale)
        else:
            st, match, _ = tempcache_merge(st, k, v, kc, F, n_f, first_frame, tau)
            if dense[s]:
                qc = np.zeros((H, 1, np.asarray(q).shape[1]), np.uint32)
                view = dataclasses.replace(st, codes=np.zeros((H, 1, st.C), np.uint32))
                o_sa, lse = annsa_attention(q, qc, view, scale)
            else:
                o_sa, lse = annsa_attention(q, qc, st, scale)
        outs.append((o_sa, lse, o_ca))
    return outs, st, match


# ---------------------------------------------------------------- quantised ANN
# The pages' other matcher ([PL] section 5 "ANN Attention": keep the keys
# with the largest query-key products, found by LSH or by quantised
# similarity search without offline preprocessing; [RB] reproduction: FAISS,
# 8-bit quantisation by default; [PL] appendix C: 2-bit to 32-bit).
# Readings: uniform scalar quantisation per dimension with `bits` bits, its
# range the minimum and maximum of the vectors being searched (nothing is
# trained offline); approximate scores use the decoded vectors; a query
# keeps the k keys of largest approximate score (ties: lower index) and
# attends them exactly (stored keys and values, + ln m); the TempCache
# matcher takes the candidate of largest approximate cosine and merges iff
# its exact cosine reaches tau.

def sq_range(x):
    """Per-dimension (lo, hi) of the rows of x [N][D]."""
    x = np.asarray(x, dtype=np.float64)
    return x.min(axis=0), x.max(axis=0)


def sq_encode(x, lo, hi, bits: int):
    """Codes in [0, 2^bits - 1]: round((x - lo) / (hi - lo) * (2^bits - 1)),
    half away from zero; a dimension with hi == lo codes to 0."""
    L = float((1 << bits) - 1)
    x = np.asarray(x, dtype=np.float64)
    span = np.asarray(hi, dtype=np.float64) - np.asarray(lo, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = np.where(span > 0, (x - lo) / np.where(span > 0, span, 1.0), 0.0)
    return np.clip(np.floor(u * L + 0.5), 0, L).astype(np.int64)


def sq_decode(c, lo, hi, bits: int):
    """The decoded vector lo + c (hi - lo) / (2^bits - 1)."""
    L = float((1 << bits) - 1)
    return np.asarray(lo, dtype=np.float64) + np.asarray(c, dtype=np.float64) * \
        (np.asarray(hi, dtype=np.float64) - np.asarray(lo, dtype=np.float64)) / L


def quant_topk(q, keys, bias, k: int, bits: int, scale: float):
    """allowed [n][M]: per query the k keys of largest approximate score
    scale q . decode(encode(key)) + bias (ties: lower index)."""
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    n, M = q.shape[0], keys.shape[0]
    allowed = np.zeros((n, M), dtype=bool)
    if M == 0 or k <= 0:
        return allowed
    lo, hi = sq_range(keys)
    xt = sq_decode(sq_encode(keys, lo, hi, bits), lo, hi, bits)
    s = scale * (q @ xt.T) + np.asarray(bias, dtype=np.float64)[None, :]
    order = np.lexsort((np.broadcast_to(np.arange(M), s.shape), -s), axis=1)[:, :min(k, M)]
    np.put_along_axis(allowed, order, True, axis=1)
    return allowed


QUANT_MARGIN = 1e-4   # score gap, relative to the vector norms, below which a selection is listed


def quant_topk_listed(q, keys, bias, k: int, bits: int, scale: float):
    """quant_topk with its near-boundary keys: (allowed [n][M], listed [n][M]).

    For query i the selection boundary is its k-th largest approximate score
    thr_i.  When two or more keys score within eps_i = QUANT_MARGIN * scale *
    |q_i| * max_s |decoded key s| of thr_i, those keys are listed: any of
    them may be the one kept (another implementation's rounding decides), so
    a comparison accepts either side for them.  Otherwise nothing is listed."""
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    n, M = q.shape[0], keys.shape[0]
    allowed = quant_topk(q, keys, bias, k, bits, scale)
    listed = np.zeros((n, M), dtype=bool)
    if M == 0 or k <= 0 or k >= M:
        return allowed, listed
    lo, hi = sq_range(keys)
    xt = sq_decode(sq_encode(keys, lo, hi, bits), lo, hi, bits)
    s = scale * (q @ xt.T) + np.asarray(bias, dtype=np.float64)[None, :]
    thr = np.partition(s, M - k, axis=1)[:, M - k]          # the k-th largest
    eps = QUANT_MARGIN * scale * np.linalg.norm(q, axis=1) * np.linalg.norm(xt, axis=1).max()
    near = np.abs(s - thr[:, None]) < eps[:, None]
    several = near.sum(axis=1) >= 2
    listed[several] = near[several]
    return allowed, listed


def annsa_quant_attention(q, state: CacheState, k: int, bits: int, scale: float):
    """AnnSA with the quantised matcher: per query the k live slots of largest
    approximate logit, attended exactly.  Returns (o, lse)."""
    q = np.asarray(q, dtype=np.float64)
    H, Nq, D = q.shape
    o = np.zeros((H, Nq, D))
    lse = np.zeros((H, Nq))
    for h in range(H):
        size = int(state.size[h])
        bias = np.log(np.maximum(state.m[h, :size], 1).astype(np.float64))
        allowed = quant_topk(q[h], state.K[h, :size], bias, k, bits, scale)
        o[h], lse[h] = masked_attention(q[h], state.K[h, :size], state.V[h, :size], allowed, bias, scale)
    return o, lse


def annca_quant_attention(q, k_p, v_p, k: int, bits: int, scale: float):
    """AnnCA with the quantised matcher: per query the k prompt tokens of
    largest approximate score, attended exactly.  Returns o."""
    q = np.asarray(q, dtype=np.float64)
    H, Nq, D = q.shape
    o = np.zeros((H, Nq, np.asarray(v_p).shape[2]))
    for h in range(H):
        P = np.asarray(k_p).shape[1]
        allowed = quant_topk(q[h], k_p[h], np.zeros(P), k, bits, scale)
        o[h], _ = masked_attention(q[h], k_p[h], v_p[h], allowed, np.zeros(P), scale)
    return o


def tempcache_nn_quant_listed(state: CacheState, k: np.ndarray, f: int, tau: float, bits: int):
    """tempcache_nn_quant with its near-boundary decisions: (match, listed).
    A decision is listed when the two best approximate cosines are within
    QUANT_MARGIN (either candidate may be taken), or when the exact cosine
    of the approximate best is within QUANT_MARGIN of tau."""
    k = np.asarray(k, dtype=np.float64)
    H, n, D = k.shape
    match = tempcache_nn_quant(state, k, f, tau, bits)
    listed = np.zeros((H, n), dtype=bool)
    for h in range(H):
        size = int(state.size[h])
        cand = np.nonzero(state.last_frame[h, :size] == f - 1)[0]
        if cand.size == 0:
            continue
        Kc = state.K[h, cand]
        lo, hi = sq_range(Kc)
        Kt = sq_decode(sq_encode(Kc, lo, hi, bits), lo, hi, bits)
        kn = np.linalg.norm(k[h], axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            approx = (k[h] @ Kt.T) / (kn[:, None] * np.linalg.norm(Kt, axis=1)[None, :])
            exact = (k[h] @ Kc.T) / (kn[:, None] * np.linalg.norm(Kc, axis=1)[None, :])
        approx[~np.isfinite(approx)] = -np.inf
        best = np.argmax(approx, axis=1)
        ex = exact[np.arange(n), best]
        near_tau = np.isfinite(ex) & (np.abs(ex - tau) < QUANT_MARGIN)
        if cand.size > 1:
            top2 = np.partition(approx, cand.size - 2, axis=1)
            with np.errstate(invalid="ignore"):
                near_tie = np.isfinite(top2[:, -1]) & ((top2[:, -1] - top2[:, -2]) < QUANT_MARGIN)
        else:
            near_tie = np.zeros(n, dtype=bool)
        listed[h] = near_tau | near_tie
    return match, listed


def tempcache_nn_quant(state: CacheState, k: np.ndarray, f: int, tau: float, bits: int):
    """TempCache's top-1 correspondence with the quantised matcher: the
    candidate (slot refreshed in frame f-1) of largest cosine between the new
    key and the candidate's decoded key (ties: lowest slot), merged iff the
    exact cosine reaches tau.  Returns match [H][n] (slot or -1)."""
    k = np.asarray(k, dtype=np.float64)
    H, n, D = k.shape
    match = np.full((H, n), -1, dtype=np.int64)
    for h in range(H):
        size = int(state.size[h])
        cand = np.nonzero(state.last_frame[h, :size] == f - 1)[0]
        if cand.size == 0:
            continue
        Kc = state.K[h, cand]
        lo, hi = sq_range(Kc)
        Kt = sq_decode(sq_encode(Kc, lo, hi, bits), lo, hi, bits)
        kn = np.linalg.norm(k[h], axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            approx = (k[h] @ Kt.T) / (kn[:, None] * np.linalg.norm(Kt, axis=1)[None, :])
            exact = (k[h] @ Kc.T) / (kn[:, None] * np.linalg.norm(Kc, axis=1)[None, :])
        approx[~np.isfinite(approx)] = -np.inf
        best = np.argmax(approx, axis=1)
        ex = exact[np.arange(n), best]
        ok = np.isfinite(approx[np.arange(n), best]) & (ex >= tau)
        match[h, ok] = cand[best[ok]]
    return match


# ---------------------------------------------------------------- recall / density
# The pages measure how much of the dense attention the sparse selections
# keep (recall and density: FAST-AR summary, paperlayer.ai section 7 and
# appendix tables; gist.science technical summary, results).  Our synthetic
# counterpart, per query i:
#   retained_i = sum_{j allowed} w_ij / sum_j w_ij,  w_ij = exp(logit_ij),
# with the same logits as the attention (AnnSA: scale q.K[s] + ln m[s] over
# the live cache; AnnCA: scale q.k_p over the prompt), i.e. the share of the
# dense softmax mass that the allowed keys carry.  Density is the allowed
# share of the (query, key) pairs.

def retained_mass(q, k, allowed, bias, scale: float):
    """Per query: the share of the dense softmax weight on its allowed keys.

    q: [n][D], k: [M][D], allowed: [n][M] bool, bias: [M].  fp64 weights
    relative to each row's dense maximum; a row of M = 0 keys gives 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if k.shape[0] == 0:
        return np.zeros(q.shape[0])
    s = scale * (q @ k.T) + np.asarray(bias, dtype=np.float64)[None, :]
    w = np.exp(s - np.max(s, axis=1, keepdims=True))
    return np.sum(np.where(allowed, w, 0.0), axis=1) / np.sum(w, axis=1)


def annsa_retained(q, q_codes, state: "CacheState", scale: float, rows=None):
    """AnnSA: (retained [H][n], density [H]) over the live cache."""
    q = np.asarray(q, dtype=np.float64)
    H, Nq, _ = q.shape
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    ret = np.zeros((H, rows.size))
    dens = np.zeros(H)
    for h in range(H):
        size = int(state.size[h])
        allowed = annsa_allowed(np.asarray(q_codes)[h][:, rows], state.codes[h, :, :size])
        bias = np.log(state.m[h, :size].astype(np.float64))
        ret[h] = retained_mass(q[h, rows], state.K[h, :size], allowed, bias, scale)
        dens[h] = allowed.mean() if allowed.size else 0.0
    return ret, dens


def annca_retained(q, k_p, kept_idx, kept_cnt, F: int, n_f: int, scale: float):
    """AnnCA: (retained [H][F*n_f], kept share [H][F]) over the prompt."""
    q = np.asarray(q, dtype=np.float64)
    H, Nq, _ = q.shape
    P = np.asarray(k_p).shape[1]
    ret = np.zeros((H, Nq))
    share = np.zeros((H, F))
    for h in range(H):
        for f in range(F):
            keep = np.zeros(P, dtype=bool)
            keep[np.asarray(kept_idx[h, f, :kept_cnt[h, f]], dtype=np.int64)] = True
            sl = slice(f * n_f, (f + 1) * n_f)
            allowed = np.broadcast_to(keep[None, :], (n_f, P))
            ret[h, sl] = retained_mass(q[h, sl], np.asarray(k_p)[h], allowed, np.zeros(P), scale)
            share[h, f] = keep.mean() if P else 0.0
    return ret, share
