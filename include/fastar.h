/*
 * fastar.h -- C ABI of the FAST-AR per-chunk attention path on GB300 (sm_103a).
 *
 * FAST-AR ("Fast Autoregressive Video Diffusion and World Models with
 * Temporal Cache Compression and Sparse Attention", arXiv 2602.01801) runs
 * three training-free modules on every generated chunk of an autoregressive
 * video diffusion model, all on one shared LSH encoding:
 *   TempCache  merge near-duplicate cached keys across frames into groups
 *              (newest key, count-weighted mean value, count m) and attend
 *              with a + ln m logit bias (exact by Lemma 5.1);
 *   AnnCA      drop prompt tokens that share no LSH bucket with a query of
 *              the current frame, then cross-attend over the survivors;
 *   AnnSA      self-attention of the chunk's queries over the merged cache,
 *              each query restricted to keys sharing one of its buckets.
 * The calls below follow that order: fastar_hash (queries, new keys, prompt
 * keys), fastar_tempcache_merge, fastar_annca_prune, fastar_annca_attention,
 * fastar_annsa_attention.
 *
 * Conventions shared by every call
 *   - Every tensor pointer is caller-owned DEVICE memory, row-major with the
 *     last dimension contiguous; rows of x/q/k/v are 16-byte aligned.
 *   - The library never allocates, frees or synchronises.  Scratch memory
 *     is the caller's workspace `ws` of at least fastar_workspace_size()
 *     bytes (256-byte aligned); it may be NULL when that size is 0.
 *   - Every call is asynchronous on `stream` and keeps no state between
 *     calls, so independent calls on different streams may run at once.
 *   - Host-detectable problems are returned as a fastar_status and nothing
 *     is launched.  Problems found on the device are written to the
 *     caller's `dev_status` word (int32, device memory, initialised to 0 by
 *     the caller): the first error wins, the library never clears it, and
 *     every later kernel that sees a non-zero status exits without writing
 *     its outputs.  No kernel traps.
 */
#ifndef FASTAR_H_
#define FASTAR_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element type of x, q, k, v, planes, the cache K/V and the outputs */
typedef enum { FASTAR_BF16 = 0, FASTAR_F32 = 1 } fastar_dtype;

typedef enum {
  FASTAR_OK = 0,
  FASTAR_ERR_ARG = 1,          /* null pointer, bad size, misaligned row     */
  FASTAR_ERR_UNSUPPORTED = 2,  /* D not in {64,128}, B > 12, T*B > 64, ...   */
  FASTAR_ERR_CUDA = 3,         /* a launch failed                            */
  FASTAR_ERR_WORKSPACE = 4,    /* ws smaller than fastar_workspace_size()   */
  FASTAR_ERR_CAPACITY = 16,    /* device: cache cannot take a frame's keys   */
  FASTAR_ERR_TIMEOUT = 17,     /* device: a bounded wait ran out             */
  FASTAR_ERR_DEVICE_ARG = 18   /* device: an index read on the device is out of range */
} fastar_status;

typedef enum {
  FASTAR_OP_HASH = 0,
  FASTAR_OP_MERGE = 1,
  FASTAR_OP_PRUNE = 2,
  FASTAR_OP_ANNCA = 3,
  FASTAR_OP_ANNSA = 4
} fastar_op;

/* Human-readable name of a fastar_status value (static string). */
const char* fastar_status_string(int status);

/* Version of this ABI (major*10000 + minor*100 + patch). */
int fastar_version(void);

/* Number of kernels this library has launched in this process (all
 * devices and threads; a diagnostic, e.g. to count launches per step). */
uint64_t fastar_launch_count(void);

/* Per-kernel launch timing (a diagnostic).  fastar_timing_begin hands the
 * library `capacity` events the caller created (cudaEventCreate, timing
 * enabled); until fastar_timing_end, the library records the next unused
 * event on the launch stream right after each kernel it launches, so the
 * time between consecutive events of one stream is the duration of the
 * kernel in between (the caller records its own event before the first
 * call).  fastar_timing_end stops recording and returns how many events were
 * recorded; fastar_timing_name(i) names the kernel that event i follows
 * (a static string; "" out of range).  Timing is process-wide: use it from
 * one thread.  NULL/0 disables it.  The library allocates nothing for it. */
int fastar_timing_begin(cudaEvent_t* events, int capacity);
int fastar_timing_end(void);
const char* fastar_timing_name(int i);

/* Self-check of the device error path (a diagnostic; the paper has no
 * counterpart).  Every mbarrier wait in this library's tensor-core kernels
 * is bounded: when it runs out the kernel writes FASTAR_ERR_TIMEOUT into
 * the caller's sticky status word, frees the TMEM it holds and returns, so
 * that the context stays usable and every later kernel of the library that
 * is given the same word exits without writing its outputs.  This call
 * launches one small kernel that allocates TMEM and waits, with that same
 * bounded wait but `polls` polls (1..FASTAR_CHECK_WAIT_MAX_POLLS, each at
 * most about 2 us), on a barrier that nothing arrives on; afterwards
 * *dev_status holds FASTAR_ERR_TIMEOUT (or the error already there).
 * Asynchronous on `stream`; FASTAR_ERR_ARG for a null word or polls out of
 * range. */
#define FASTAR_CHECK_WAIT_MAX_POLLS 65536
int fastar_check_bounded_wait(int polls, int32_t* dev_status, cudaStream_t stream);

/*
 * Bytes of workspace a call needs.  Arguments that an op does not use are
 * ignored.  op: FASTAR_OP_*; H heads; N rows per head (hash: N; merge:
 * n_f, the tokens per frame; prune: P; annca: F, the frames of the chunk;
 * annsa: Nq); D head dim; T tables; B bits; C cache capacity (annca: P, the
 * prompt tokens).
 */
size_t fastar_workspace_size(int op, int H, int N, int D, int T, int B, int C);

/*
 * fastar_hash -- random-hyperplane LSH codes, optionally with bucket CSR.
 *
 * Passage: FAST-AR summary (paperlayer.ai) section 2, approximate nearest
 * neighbour search (LSH with multi-table bucket probing) and section 5
 * "ANN Attention"; FAST-AR technical summary (gist.science) 2.B (queries
 * and prompt keys projected into one shared LSH space); FAST-AR analysis
 * (paper.rainbus.top), technical novelty (the hash is computed once and
 * serves all three modules).
 *
 *   codes[h][t][i] = sum_{b<B} [ planes[t*B+b] . x[h][i] > 0 ] << b
 *
 * x       [H][N][D] dt     rows to hash (queries, new keys or prompt keys)
 * planes  [T*B][D]  dt     hyperplanes, shared by every head and every caller
 * codes   [H][T][N] uint32 output
 * perm    [H][T][N] int32  optional (NULL): ids 0..N-1 grouped by code,
 *                          stable (ascending id inside a bucket)
 * offsets [H][T][2^B+1] int32 optional, with perm: offsets[c] = number of
 *                          ids whose code is < c
 * Limits: D in {64, 128}; 1 <= T*B <= 64; B <= 12 when perm is requested.
 * Products are exact in fp32 and accumulated in fp32; a bit whose
 * projection is within fp32 rounding of 0 may take either value.
 */
int fastar_hash(fastar_dtype dt, const void* x, int H, int N, int D,
                const void* planes, int T, int B, uint32_t* codes,
                int32_t* perm, int32_t* offsets, void* ws, size_t ws_bytes,
                int32_t* dev_status, cudaStream_t stream);

/*
 * fastar_bucket_csr -- the bucket CSR of fastar_hash (perm / offsets) for
 * codes that are already there: per group g (a head and table), a stable
 * counting sort of the ids 0..N-1 by code.  Same passage as fastar_hash (the
 * buckets of each LSH table).
 *
 * codes   [G][N] uint32, every value < 2^B (FASTAR_ERR_DEVICE_ARG otherwise)
 * perm    [G][N] int32   ids grouped by code, ascending id inside a bucket
 * offsets [G][2^B+1] int32 offsets[c] = number of ids whose code is < c
 * Limits: B <= 12.
 */
int fastar_bucket_csr(const uint32_t* codes, int G, int N, int B, int32_t* perm,
                      int32_t* offsets, int32_t* dev_status, cudaStream_t stream);

/*
 * fastar_hash_many -- the same codes (and optional bucket CSR) for up to
 * FASTAR_MAX_HASH_JOBS inputs that share H, D, the hyperplanes, T and B, in
 * one pass: the result equals one fastar_hash call per job, in job order.
 * The chunk path hashes its queries, new keys and prompt keys this way (the
 * hash is computed once and serves all three modules; same passages as
 * fastar_hash).
 *
 * jobs    host array of n_jobs entries (1 <= n_jobs <= FASTAR_MAX_HASH_JOBS),
 *         read during the call only; job j: x [H][N][D] dt, codes
 *         [H][T][N], optional perm / offsets as for fastar_hash.  A job with
 *         N == 0 is skipped.
 * Errors as for fastar_hash; FASTAR_ERR_ARG for a bad n_jobs or job.
 */
#define FASTAR_MAX_HASH_JOBS 4
typedef struct fastar_hash_job {
  const void* x;
  int N;
  uint32_t* codes;
  int32_t* perm;
  int32_t* offsets;
} fastar_hash_job;

int fastar_hash_many(fastar_dtype dt, int n_jobs, const fastar_hash_job* jobs,
                     int H, int D, const void* planes, int T, int B,
                     void* ws, size_t ws_bytes, int32_t* dev_status,
                     cudaStream_t stream);

/*
 * The merged cache of one layer: fixed capacity C per head, all buffers
 * caller-owned device memory, allocated once.  Initialise last_frame to -1
 * and every other buffer to 0.  Checkpointing the cache means copying
 * these buffers.
 *   K, V        [H][C][D] dt   representative key / mean value of a group
 *   m           [H][C] int32   group count (multiplicity)
 *   codes       [H][T][C] uint32 LSH codes of K
 *   last_frame  [H][C] int32   frame that last refreshed the group, -1 empty
 *   size        [H] int32      live slots; slots >= size are empty
 *   inserted    [H] int64      keys ever merged in
 *   evicted     [H] int64      sum of m over evicted groups
 *   perm        [H][T][C] int32  CSR of the live codes (first size entries)
 *   offsets     [H][T][2^B+1] int32
 * Invariant: sum of m over live slots + evicted == inserted.
 */
typedef struct {
  int H, D, C, T, B;
  fastar_dtype dt;
  void* K;
  void* V;
  int32_t* m;
  uint32_t* codes;
  int32_t* last_frame;
  int32_t* size;
  int64_t* inserted;
  int64_t* evicted;
  int32_t* perm;
  int32_t* offsets;
} fastar_cache;

/*
 * fastar_tempcache_merge -- merge the F frames of a chunk into the cache.
 *
 * Passage: FAST-AR summary (paperlayer.ai) section 5 "TempCache" (top-1
 * ANN correspondence, recent representatives, mean values and + log m_t)
 * and appendix A (Lemma A.1); FAST-AR technical summary (gist.science) 2.A
 * (merging bounds the cache, so memory and latency stay constant); FAST-AR
 * analysis (paper.rainbus.top), method steps, TempCache.
 *
 * Frame f = first_frame + i (i = 0..F-1) is merged after frame f-1:
 *   1. every key k_j of frame f is matched to the live group s with
 *      last_frame[s] == f-1 of largest cosine(k_j, K[s]) (ties: lowest s);
 *      it joins s iff that cosine >= tau;
 *   2. a group joined by the keys S gets m' = m + |S|,
 *      V' = (m V + sum_{j in S} v_j) / m' (fp32, rounded to dt), and K,
 *      codes and last_frame of the lowest j in S;
 *   3. unmatched keys (ascending j) become groups of count 1 in the free
 *      slots size, size+1, ... and then in evicted slots: the groups with
 *      the smallest (last_frame, slot) among those with last_frame < f, in
 *      ascending slot order; evicted += their m; inserted += n_f.
 * Afterwards the CSR (perm, offsets) of the live codes is rebuilt.
 *
 * k_new, v_new [H][F*n_f][D] dt; codes_new [H][T][F*n_f] uint32 (from
 * fastar_hash of k_new with the cache's planes); match_out optional
 * [H][F*n_f] int32: the slot each key joined, or -1.
 * Requires n_f <= C (then step 3 always finds room) and
 * n_f <= FASTAR_MAX_FRAME_KEYS (FASTAR_ERR_UNSUPPORTED otherwise).
 */
int fastar_tempcache_merge(const fastar_cache* cache, const void* k_new,
                           const void* v_new, const uint32_t* codes_new,
                           int F, int n_f, int32_t first_frame, float tau,
                           int32_t* match_out, void* ws, size_t ws_bytes,
                           int32_t* dev_status, cudaStream_t stream);

/* Largest frame (keys per frame) the merge accepts: the per-frame plan keeps
 * each key's match and a hash table of the frame's groups in shared memory. */
#define FASTAR_MAX_FRAME_KEYS 6144

/*
 * fastar_tempcache_merge_ev -- fastar_tempcache_merge whose codes_new (and
 * v_new) may still be in the making when the call is issued: codes_ready
 * (an event recorded after the work that writes them, typically on another
 * stream; NULL: none) is waited on by `stream` right before the first
 * kernel that reads codes_new or v_new.  The candidate setup, the first
 * frame's nearest-neighbour search and its plan, which read only k_new and
 * the cache, run before that wait, so a caller can hash the chunk on
 * another stream meanwhile.  k_new must be ready on `stream` as usual.
 * Same arguments, results and errors otherwise.
 */
int fastar_tempcache_merge_ev(const fastar_cache* cache, const void* k_new,
                              const void* v_new, const uint32_t* codes_new,
                              int F, int n_f, int32_t first_frame, float tau,
                              int32_t* match_out, void* ws, size_t ws_bytes,
                              int32_t* dev_status, cudaStream_t stream,
                              cudaEvent_t codes_ready);

/*
 * fastar_tempcache_merge_rep -- fastar_tempcache_merge_ev with a choice of
 * the group representative.
 *
 * Passage: FAST-AR summary (paperlayer.ai) appendix C, representative
 * selection in KV merging (last-key, mean-key and medoid-key
 * representatives of a group of corresponding keys; the method keeps the
 * last key).
 *
 * rep = FASTAR_REP_LAST: exactly fastar_tempcache_merge_ev (planes may be
 * NULL).  rep = FASTAR_REP_MEAN: step 2 keeps the count-weighted mean key
 * instead of the lowest j's key, K' = (m K + sum_{j in S} k_j) / m' (fp32,
 * rounded to dt like V), and the group's codes become the hash of the stored
 * K' with `planes` [T*B][D] dt (the hyperplanes codes_new came from; bits as
 * in fastar_hash, a zero projection gives 0).  Unmatched keys are inserted
 * as in the last-key mode.  The next frame is matched against the stored
 * (mean) keys.  codes_ready as in fastar_tempcache_merge_ev (NULL: none).
 * Errors as fastar_tempcache_merge, plus FASTAR_ERR_ARG for an unknown rep,
 * or a NULL or misaligned planes with FASTAR_REP_MEAN; FASTAR_ERR_UNSUPPORTED
 * when T*B > 64 with FASTAR_REP_MEAN.  The medoid-key representative needs
 * every past member of a group and is not offered.
 */
#define FASTAR_REP_LAST 0
#define FASTAR_REP_MEAN 1
int fastar_tempcache_merge_rep(const fastar_cache* cache, const void* k_new,
                               const void* v_new, const uint32_t* codes_new,
                               int F, int n_f, int32_t first_frame, float tau,
                               int rep, const void* planes,
                               int32_t* match_out, void* ws, size_t ws_bytes,
                               int32_t* dev_status, cudaStream_t stream,
                               cudaEvent_t codes_ready);

/*
 * fastar_tempcache_merge_search -- fastar_tempcache_merge with a choice of
 * where step 1 looks for the nearest earlier group.
 *
 * Passage: FAST-AR technical summary (gist.science) 2.A (the nearest key
 * among the earlier frames is found with LSH or quantisation); FAST-AR
 * analysis (paper.rainbus.top), method steps, TempCache (the default looks
 * at the previous frame).
 *
 * search = FASTAR_SEARCH_PREV: exactly fastar_tempcache_merge_ev (the
 * groups refreshed in frame f-1).  search = FASTAR_SEARCH_LSH: the
 * candidates of k_j are every live group (refreshed in any earlier frame)
 * that shares an LSH bucket with k_j in some table (the cache's stored
 * codes against codes_new); largest cosine, ties to the lowest slot, joined
 * iff the cosine >= tau; step 3 never evicts a group joined in the same
 * frame.  The cache CSR (perm, offsets) is rebuilt before every frame's
 * search, so the caller's CSR need not be current; with FASTAR_SEARCH_LSH
 * codes_ready (NULL: none) is waited for before the first search.
 * search = FASTAR_SEARCH_QUANT_BITS(b), 1 <= b <= 16 (the quantised
 * matcher, TempCache-Quant; FAST-AR summary (paperlayer.ai) section 5 "ANN
 * Attention" and appendix C; paper.rainbus.top, reproduction: 8-bit codes
 * by default): the candidates are frame f-1's groups as in
 * FASTAR_SEARCH_PREV, quantised per dimension over their own range to b-bit
 * codes (code = floor((x - lo) / (hi - lo) (2^b - 1) + 0.5), computed in
 * fp64); k_j takes the candidate of largest cosine to its decoded key (ties:
 * lowest slot) and joins it iff the exact cosine reaches tau.  bf16 with
 * D = 128 only (FASTAR_ERR_UNSUPPORTED otherwise); a frame with more than
 * n_f candidates (left by a call with larger frames) sets
 * FASTAR_ERR_DEVICE_ARG.  Same workspace as fastar_tempcache_merge; errors
 * as fastar_tempcache_merge, plus FASTAR_ERR_ARG for an unknown search.
 */
#define FASTAR_SEARCH_PREV 0
#define FASTAR_SEARCH_LSH 1
#define FASTAR_SEARCH_QUANT 2
#define FASTAR_SEARCH_QUANT_BITS(b) (FASTAR_SEARCH_QUANT | ((b) << 8))
int fastar_tempcache_merge_search(const fastar_cache* cache, const void* k_new,
                                  const void* v_new, const uint32_t* codes_new,
                                  int F, int n_f, int32_t first_frame, float tau,
                                  int search, int32_t* match_out, void* ws,
                                  size_t ws_bytes, int32_t* dev_status,
                                  cudaStream_t stream, cudaEvent_t codes_ready);

/*
 * fastar_tempcache_merge_noalloc -- fastar_tempcache_merge without a
 * caller workspace.  The paper has no counterpart: this is a convenience of
 * this library for callers that cannot allocate device memory, such as a
 * plugin inside a host application that owns the GPU's memory budget, or a
 * C/FFI caller that holds only the pointers handed to it.
 *
 * Same arguments and results as fastar_tempcache_merge, minus ws/ws_bytes.
 * The scratch is a fixed array of FASTAR_NOALLOC_SCRATCH_BYTES inside the
 * library's device memory, held by every GPU that loads the library until
 * the process exits.  Returns FASTAR_ERR_WORKSPACE when the merge needs more
 * (fastar_workspace_size(FASTAR_OP_MERGE, ...) > FASTAR_NOALLOC_SCRATCH_BYTES;
 * e.g. 12 heads x C 32768 x n_f 1560 needs about 10 MiB and fits, 40 heads
 * x n_f 3600 needs about 56 MiB and is refused).  All calls
 * share the array, so calls that overlap on the GPU race and must be ordered
 * by the caller; it keeps the last call's contents (the merge needs none of
 * it zeroed).  The first call on a device looks up the array's address with
 * that device current; make it before any stream capture.
 */
#define FASTAR_NOALLOC_SCRATCH_BYTES (16u << 20)
int fastar_tempcache_merge_noalloc(const fastar_cache* cache, const void* k_new,
                                   const void* v_new, const uint32_t* codes_new,
                                   int F, int n_f, int32_t first_frame, float tau,
                                   int32_t* match_out, int32_t* dev_status,
                                   cudaStream_t stream);

/*
 * fastar_annca_prune -- per-frame prompt-token selection for AnnCA.
 *
 * Passage: FAST-AR technical summary (gist.science) 2.B AnnCA mechanism
 * (a prompt token is kept for a frame iff it shares a bucket with at least
 * one query of that frame); FAST-AR analysis (paper.rainbus.top), method
 * steps, AnnCA; FAST-AR summary (paperlayer.ai) section 5 "AnnCA".
 *
 * q_codes [H][T][F*n_f], p_codes [H][T][P] uint32 (codes < 2^B).
 * kept_idx [H][F][P] int32: ascending kept prompt ids of (head, frame),
 * padded with -1; kept_cnt [H][F] int32.  Multi-table = union over tables.
 */
int fastar_annca_prune(const uint32_t* q_codes, const uint32_t* p_codes,
                       int H, int F, int n_f, int P, int T, int B,
                       int32_t* kept_idx, int32_t* kept_cnt, void* ws,
                       size_t ws_bytes, int32_t* dev_status, cudaStream_t stream);

/*
 * fastar_annca_attention -- cross-attention over the kept prompt tokens.
 *
 * Passage: FAST-AR technical summary (gist.science) 2.B; FAST-AR summary
 * (paperlayer.ai) section 3, attention formulation (cross-attention keys are
 * the projected prompt tokens).
 *
 *   out[h][i] = sum_{p in kept(h, i / n_f)} softmax_p(scale q_i.k_p) v_p
 *   (0 when the kept set is empty)
 *
 * q [H][F*n_f][D], k_p, v_p [H][P][D] dt; kept_idx/kept_cnt from
 * fastar_annca_prune (or any ascending id list); out [H][F*n_f][D] dt.
 * ws: fastar_workspace_size(FASTAR_OP_ANNCA, H, F, D, 0, 0, P) bytes (the
 * kept rows of each frame are compacted there; FASTAR_ERR_WORKSPACE when
 * smaller).  scale must be positive and finite (FASTAR_ERR_ARG otherwise).
 * fp32 accumulation.  Passing kept = 0..P-1 gives dense attention.
 */
int fastar_annca_attention(fastar_dtype dt, const void* q, const void* k_p,
                           const void* v_p, const int32_t* kept_idx,
                           const int32_t* kept_cnt, int H, int F, int n_f,
                           int P, int D, float scale, void* out, void* ws,
                           size_t ws_bytes, int32_t* dev_status,
                           cudaStream_t stream);

/*
 * fastar_annsa_attention -- bucket-restricted self-attention over the cache.
 *
 * Passage: FAST-AR technical summary (gist.science) 2.C (each query attends
 * only keys in its own semantic bucket(s)); FAST-AR analysis
 * (paper.rainbus.top), method steps, AnnSA; FAST-AR summary (paperlayer.ai)
 * appendix A, Lemma A.1 (+ log m_t bias of merged groups).
 *
 *   allowed(i, s) <=> s < size and exists t: q_codes[t][i] == codes[t][s]
 *   out[h][i] = sum_{allowed s} softmax_s(scale q_i.K[s] + ln m[s]) V[s]
 *   lse[h][i] = ln sum_{allowed s} exp(scale q_i.K[s] + ln m[s])
 *   (out = 0 and lse = -inf when nothing is allowed)
 *
 * q [H][Nq][D] dt; q_codes [H][T][Nq]; q_perm [H][T][Nq] and q_offsets
 * [H][T][2^B+1] from fastar_hash of q; the cache after the chunk's merge;
 * out [H][Nq][D] dt; lse optional [H][Nq] float.  scale must be positive
 * and finite (FASTAR_ERR_ARG otherwise).  fp32 accumulation.
 */
int fastar_annsa_attention(fastar_dtype dt, const void* q,
                           const uint32_t* q_codes, const int32_t* q_perm,
                           const int32_t* q_offsets, int Nq,
                           const fastar_cache* cache, float scale, void* out,
                           float* lse, void* ws, size_t ws_bytes,
                           int32_t* dev_status, cudaStream_t stream);

/*
 * fastar_annsa_attention_part / fastar_annsa_combine -- AnnSA over several
 * key sets whose results are merged exactly, for the denoising steps of a
 * chunk.
 *
 * Passage: FAST-AR analysis (paper.rainbus.top), limitations (sparse
 * attention is off for the first 30 % of the denoising steps) and method
 * steps, AnnSA; FAST-AR summary (paperlayer.ai) related work (each chunk is
 * denoised conditioned on the history).  A denoising step before the last
 * attends the cache together with its own keys, which are not merged into
 * it: the caller describes those keys as a second fastar_cache (K, V = the
 * step's keys and values, m = 1, codes and CSR of their hash, size = Nq)
 * and, for a dense step, both key sets with one table of one bit whose codes
 * are all 0 (every pair allowed).
 *
 * fastar_annsa_attention_part computes what fastar_annsa_attention does
 * for `cache`, but leaves each table's partial (its output normalised by its
 * own sum, in fp16, with its max and sum in fp32) in slots part_base ..
 * part_base + T - 1 of a workspace of part_total
 * slots (sized by fastar_workspace_size(FASTAR_OP_ANNSA_PARTS, H, Nq, D,
 * part_total, ...)); nothing else is written.  fastar_annsa_combine then
 * merges the part_total partials of every query (the softmax over the union
 * of the key sets, which must be disjoint) into out [H][Nq][D] dt and the
 * optional lse [H][Nq].  1 <= part_total <= 4 and part_base + T <=
 * part_total (FASTAR_ERR_ARG otherwise); bf16 with D = 128 only
 * (FASTAR_ERR_UNSUPPORTED otherwise).  Every slot must be written by a part
 * call on the same stream before the combine.
 */
#define FASTAR_OP_ANNSA_PARTS 5
int fastar_annsa_attention_part(fastar_dtype dt, const void* q,
                                const uint32_t* q_codes, const int32_t* q_perm,
                                const int32_t* q_offsets, int Nq,
                                const fastar_cache* cache, float scale,
                                int part_base, int part_total, void* ws,
                                size_t ws_bytes, int32_t* dev_status,
                                cudaStream_t stream);
int fastar_annsa_combine(int H, int Nq, int D, int part_total, const void* ws,
                         size_t ws_bytes, void* out, float* lse,
                         int32_t* dev_status, cudaStream_t stream);

/*
 * fastar_annsa_quant_attention / fastar_annca_quant_attention -- AnnSA and
 * AnnCA with the quantised matcher instead of the LSH buckets.
 *
 * Passage: FAST-AR summary (paperlayer.ai) section 5 "ANN Attention" (keep
 * the keys of largest query-key product, found by LSH or by quantised
 * similarity search without offline preprocessing) and appendix C
 * (quantisation precision for ANN matching, 2 to 32 bits); FAST-AR analysis
 * (paper.rainbus.top), reproduction (FAISS, 8-bit by default).
 *
 * The keys of each head (AnnSA: the live cache slots; AnnCA: the P prompt
 * tokens) are quantised per dimension over their own range [lo, hi] to
 * `bits`-bit codes, code = floor((x - lo) / (hi - lo) (2^bits - 1) + 0.5)
 * (0 where hi == lo; computed in fp64), decoded as lo + code (hi - lo) /
 * (2^bits - 1).  Each query keeps the topk keys of largest approximate
 * score scale q . decoded + bias (AnnSA: bias ln m; AnnCA: 0; ties: lower
 * index; every key when topk >= their number) and attends them exactly:
 *   out[h][i] = sum_{kept s} softmax_s(scale q_i.K[s] + bias_s) V[s]
 * (lse as for fastar_annsa_attention).  sel_mask, optional [H][Nq][ceil(N /
 * 32)] uint32 (N = C or P), receives the kept keys as bits (bit s % 32 of
 * word s / 32).  bf16 with D = 128; 1 <= bits <= 16 (FASTAR_ERR_UNSUPPORTED
 * otherwise).  ws: fastar_workspace_size(FASTAR_OP_QUANT, H, Nq, D, bits, 0,
 * N) bytes (codes, scores of a batch of heads, the selection).  Approximate
 * scores are fp32; keys whose score is within rounding of the topk-th may
 * fall on either side.  Errors as fastar_annsa_attention.
 */
#define FASTAR_OP_QUANT 6
int fastar_annsa_quant_attention(fastar_dtype dt, const void* q, int Nq,
                                 const fastar_cache* cache, float scale, int topk,
                                 int bits, void* out, float* lse, uint32_t* sel_mask,
                                 void* ws, size_t ws_bytes, int32_t* dev_status,
                                 cudaStream_t stream);
int fastar_annca_quant_attention(fastar_dtype dt, const void* q, const void* k_p,
                                 const void* v_p, int H, int Nq, int P, int D,
                                 float scale, int topk, int bits, void* out,
                                 uint32_t* sel_mask, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FASTAR_H_ */
