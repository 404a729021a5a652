// C ABI of the FAST-AR per-chunk attention path: argument checks, workspace
// sizing and dispatch to the kernels.  Nothing here allocates, frees or
// synchronises; every launch goes to the caller's stream.
#include <string.h>

#include <atomic>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"

namespace fastar {
// Every compute call is an NVTX range named after it, so that a profiler's
// timeline shows which call launched which kernels (a no-op without one).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
static std::atomic<uint64_t> g_launches{0};

// launch timing: caller-created events, recorded after each launch
static std::mutex g_tmu;
static std::atomic<int> g_timing{0};
static cudaEvent_t* g_tev = nullptr;
static int g_tcap = 0, g_tn = 0;
static const char* g_tname[4096];

void after_launch(cudaStream_t s, const char* name) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_timing.load(std::memory_order_acquire)) return;
  std::lock_guard<std::mutex> lock(g_tmu);
  if (g_tev && g_tn < g_tcap && g_tn < 4096) {
    if (cudaEventRecord(g_tev[g_tn], s) == cudaSuccess) g_tname[g_tn++] = name;
    else (void)cudaGetLastError();
  }
}

int launch_hash_simt(fastar_dtype dt, const void* x, int H, int N, int D, const void* planes,
                     int T, int B, uint32_t* codes, int32_t* st, cudaStream_t s);
int launch_hash_tc(fastar_dtype dt, const void* x, int H, int N, int D, const void* planes,
                   int T, int B, uint32_t* codes, int32_t* st, cudaStream_t s);
int launch_hash_tc_many(fastar_dtype dt, int n, const void* const* xs, const int* Ns, uint32_t* const* codes,
                        int H, int D, const void* planes, int T, int B, int32_t* st, cudaStream_t s);
int launch_annca_simt(fastar_dtype dt, const void* q, const void* k_p, const void* v_p,
                      const int32_t* kept_idx, const int32_t* kept_cnt, int H, int F, int n_f, int P,
                      int D, float scale, void* out, int32_t* st, cudaStream_t s);
int launch_annca_tc(fastar_dtype dt, const void* q, const void* k_p, const void* v_p,
                    const int32_t* kept_idx, const int32_t* kept_cnt, int H, int F, int n_f, int P,
                    int D, float scale, void* out, void* ws, size_t ws_bytes, int32_t* st, cudaStream_t s);
size_t annca_tc_ws_bytes(int H, int F, int P, int D);
int launch_annsa_simt(fastar_dtype dt, const void* q, const uint32_t* q_codes, int Nq,
                      const fastar_cache* c, float scale, void* out, float* lse, int32_t* st,
                      cudaStream_t s);
int launch_annsa_tc(fastar_dtype dt, const void* q, const uint32_t* q_codes, const int32_t* q_perm,
                    const int32_t* q_offsets, int Nq, const fastar_cache* c, float scale, void* out,
                    float* lse, void* ws, int32_t* st, cudaStream_t s);
size_t annsa_tc_ws_bytes(int H, int Nq, int D, int T);
size_t annsa_parts_ws_bytes(int H, int Nq, int D, int parts);
int launch_annsa_parts(const void* q, const uint32_t* q_codes, const int32_t* q_perm, int Nq,
                       const fastar_cache* c, float scale, int base, int parts, void* ws, int32_t* st,
                       cudaStream_t s);
int launch_annsa_combine(int H, int Nq, int parts, const void* ws, void* out, float* lse, int32_t* st,
                         cudaStream_t s);

int launch_hash(fastar_dtype dt, const void* x, int H, int N, int D, const void* planes, int T,
                int B, uint32_t* codes, int32_t* st, cudaStream_t s) {
  int rc = launch_hash_tc(dt, x, H, N, D, planes, T, B, codes, st, s);
  if (rc != FASTAR_ERR_UNSUPPORTED) return rc;
  return launch_hash_simt(dt, x, H, N, D, planes, T, B, codes, st, s);
}

int launch_annca(fastar_dtype dt, const void* q, const void* k_p, const void* v_p,
                 const int32_t* kept_idx, const int32_t* kept_cnt, int H, int F, int n_f, int P,
                 int D, float scale, void* out, void* ws, size_t ws_bytes, int32_t* st, cudaStream_t s) {
  int rc = launch_annca_tc(dt, q, k_p, v_p, kept_idx, kept_cnt, H, F, n_f, P, D, scale, out, ws, ws_bytes,
                           st, s);
  if (rc != FASTAR_ERR_UNSUPPORTED) return rc;
  return launch_annca_simt(dt, q, k_p, v_p, kept_idx, kept_cnt, H, F, n_f, P, D, scale, out, st, s);
}

int launch_annsa(fastar_dtype dt, const void* q, const uint32_t* q_codes, const int32_t* q_perm,
                 const int32_t* q_offsets, int Nq, const fastar_cache* c, float scale, void* out,
                 float* lse, void* ws, int32_t* st, cudaStream_t s) {
  int rc = launch_annsa_tc(dt, q, q_codes, q_perm, q_offsets, Nq, c, scale, out, lse, ws, st, s);
  if (rc != FASTAR_ERR_UNSUPPORTED) return rc;
  return launch_annsa_simt(dt, q, q_codes, Nq, c, scale, out, lse, st, s);
}

size_t annsa_ws_bytes(int H, int Nq, int D, int T) { return annsa_tc_ws_bytes(H, Nq, D, T); }

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }
static bool dtype_ok(int dt) { return dt == FASTAR_BF16 || dt == FASTAR_F32; }
static bool dim_ok(int D) { return D == 64 || D == 128; }

}  // namespace fastar

using namespace fastar;

extern "C" {

const char* fastar_status_string(int status) {
  switch (status) {
    case FASTAR_OK: return "ok";
    case FASTAR_ERR_ARG: return "invalid argument";
    case FASTAR_ERR_UNSUPPORTED: return "unsupported shape or type";
    case FASTAR_ERR_CUDA: return "CUDA launch error";
    case FASTAR_ERR_WORKSPACE: return "workspace too small";
    case FASTAR_ERR_CAPACITY: return "cache capacity exhausted (device)";
    case FASTAR_ERR_TIMEOUT: return "bounded device wait expired (device)";
    case FASTAR_ERR_DEVICE_ARG: return "out-of-range index found on the device";
    default: return "unknown status";
  }
}

int fastar_version(void) { return 300; }

uint64_t fastar_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int fastar_timing_begin(cudaEvent_t* events, int capacity) {
  if (capacity < 0 || (capacity > 0 && !events)) return FASTAR_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_tmu);
  g_tev = events;
  g_tcap = capacity;
  g_tn = 0;
  g_timing.store(capacity > 0 ? 1 : 0, std::memory_order_release);
  return FASTAR_OK;
}

int fastar_timing_end(void) {
  std::lock_guard<std::mutex> lock(g_tmu);
  g_timing.store(0, std::memory_order_release);
  g_tev = nullptr;
  g_tcap = 0;
  return g_tn;
}

const char* fastar_timing_name(int i) {
  std::lock_guard<std::mutex> lock(g_tmu);
  return (i >= 0 && i < g_tn) ? g_tname[i] : "";
}

size_t fastar_workspace_size(int op, int H, int N, int D, int T, int B, int C) {
  (void)B;
  if (H < 0 || N < 0 || C < 0) return 0;
  switch (op) {
    case FASTAR_OP_MERGE: return merge_ws_bytes(H, N, C);
    case FASTAR_OP_ANNCA: return annca_tc_ws_bytes(H, N, C, D);  // N = frames F, C = prompt tokens P
    case FASTAR_OP_ANNSA: return annsa_ws_bytes(H, N, D, T);
    case FASTAR_OP_ANNSA_PARTS: return annsa_parts_ws_bytes(H, N, D, T);  // T = part_total
    case FASTAR_OP_QUANT: return quant_ws_bytes(H, N, C, D, T);  // N = Nq, T = bits, C = keys per head
    default: return 0;
  }
}

int fastar_hash(fastar_dtype dt, const void* x, int H, int N, int D, const void* planes, int T,
                int B, uint32_t* codes, int32_t* perm, int32_t* offsets, void* ws, size_t ws_bytes,
                int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_hash");
  (void)ws;
  (void)ws_bytes;
  if (!dtype_ok(dt)) return FASTAR_ERR_UNSUPPORTED;
  if (H < 0 || N < 0 || T < 1 || B < 1 || T > 8) return FASTAR_ERR_ARG;
  if (!dim_ok(D) || T * B > kMaxTB) return FASTAR_ERR_UNSUPPORTED;
  if ((perm == nullptr) != (offsets == nullptr)) return FASTAR_ERR_ARG;
  if (perm && B > kMaxCsrBits) return FASTAR_ERR_UNSUPPORTED;
  if ((size_t)H * N == 0) return FASTAR_OK;
  if (!x || !planes || !codes || !aligned16(x) || !aligned16(planes)) return FASTAR_ERR_ARG;
  int rc = launch_hash(dt, x, H, N, D, planes, T, B, codes, dev_status, stream);
  if (rc != FASTAR_OK || !perm) return rc;
  return launch_csr(codes, H * T, N, nullptr, 1, 1 << B, perm, offsets, dev_status, stream);
}

int fastar_bucket_csr(const uint32_t* codes, int G, int N, int B, int32_t* perm, int32_t* offsets,
                      int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_bucket_csr");
  if (G < 0 || N < 0 || B < 1) return FASTAR_ERR_ARG;
  if (B > kMaxCsrBits) return FASTAR_ERR_UNSUPPORTED;
  if ((size_t)G * N == 0) return FASTAR_OK;
  if (!codes || !perm || !offsets) return FASTAR_ERR_ARG;
  return launch_csr(codes, G, N, nullptr, 1, 1 << B, perm, offsets, dev_status, stream);
}

int fastar_hash_many(fastar_dtype dt, int n_jobs, const fastar_hash_job* jobs, int H, int D,
                     const void* planes, int T, int B, void* ws, size_t ws_bytes, int32_t* dev_status,
                     cudaStream_t stream) {
  CallRange range("fastar_hash_many");
  (void)ws;
  (void)ws_bytes;
  if (!dtype_ok(dt)) return FASTAR_ERR_UNSUPPORTED;
  if (n_jobs < 1 || n_jobs > FASTAR_MAX_HASH_JOBS || !jobs) return FASTAR_ERR_ARG;
  if (H < 0 || T < 1 || B < 1 || T > 8) return FASTAR_ERR_ARG;
  if (!dim_ok(D) || T * B > kMaxTB) return FASTAR_ERR_UNSUPPORTED;
  const void* xs[FASTAR_MAX_HASH_JOBS];
  int Ns[FASTAR_MAX_HASH_JOBS];
  uint32_t* cs[FASTAR_MAX_HASH_JOBS];
  int n = 0;
  for (int j = 0; j < n_jobs; ++j) {
    const fastar_hash_job& q = jobs[j];
    if (q.N < 0 || (q.perm == nullptr) != (q.offsets == nullptr)) return FASTAR_ERR_ARG;
    if (q.perm && B > kMaxCsrBits) return FASTAR_ERR_UNSUPPORTED;
    if ((size_t)H * q.N == 0) continue;
    if (!q.x || !q.codes || !aligned16(q.x)) return FASTAR_ERR_ARG;
    xs[n] = q.x;
    Ns[n] = q.N;
    cs[n] = q.codes;
    ++n;
  }
  if (n == 0) return FASTAR_OK;
  if (!planes || !aligned16(planes)) return FASTAR_ERR_ARG;
  int rc = launch_hash_tc_many(dt, n, xs, Ns, cs, H, D, planes, T, B, dev_status, stream);
  if (rc == FASTAR_ERR_UNSUPPORTED) {
    rc = FASTAR_OK;
    for (int j = 0; j < n && rc == FASTAR_OK; ++j)
      rc = launch_hash(dt, xs[j], H, Ns[j], D, planes, T, B, cs[j], dev_status, stream);
  }
  for (int j = 0; j < n_jobs && rc == FASTAR_OK; ++j) {
    const fastar_hash_job& q = jobs[j];
    if (q.perm && (size_t)H * q.N > 0)
      rc = launch_csr(q.codes, H * T, q.N, nullptr, 1, 1 << B, q.perm, q.offsets, dev_status, stream);
  }
  return rc;
}

static int check_cache(const fastar_cache* c) {
  if (!c) return FASTAR_ERR_ARG;
  if (!dtype_ok(c->dt)) return FASTAR_ERR_UNSUPPORTED;
  if (c->H < 0 || c->C < 1 || c->T < 1 || c->T > 8 || c->B < 1) return FASTAR_ERR_ARG;
  if (!dim_ok(c->D) || c->B > kMaxCsrBits) return FASTAR_ERR_UNSUPPORTED;
  if (!c->K || !c->V || !c->m || !c->codes || !c->last_frame || !c->size || !c->inserted ||
      !c->evicted || !c->perm || !c->offsets)
    return FASTAR_ERR_ARG;
  if (!aligned16(c->K) || !aligned16(c->V)) return FASTAR_ERR_ARG;
  return FASTAR_OK;
}

static int merge_checked(const fastar_cache* cache, const void* k_new, const void* v_new,
                         const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                         int32_t* match_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                         cudaStream_t stream, cudaEvent_t codes_ready, int rep = FASTAR_REP_LAST,
                         const void* planes = nullptr, int search = FASTAR_SEARCH_PREV) {
  int rc = check_cache(cache);
  if (rc != FASTAR_OK) return rc;
  if (rep != FASTAR_REP_LAST && rep != FASTAR_REP_MEAN) return FASTAR_ERR_ARG;
  const bool quant_ok = (search & 0xff) == FASTAR_SEARCH_QUANT && (search >> 8) >= 1 && (search >> 8) <= 16;
  if (search != FASTAR_SEARCH_PREV && search != FASTAR_SEARCH_LSH && !quant_ok) return FASTAR_ERR_ARG;
  if (rep == FASTAR_REP_MEAN) {
    if (!planes || !aligned16(planes)) return FASTAR_ERR_ARG;
    if (cache->T * cache->B > 64) return FASTAR_ERR_UNSUPPORTED;
  }
  if (F < 0 || n_f < 0 || n_f > cache->C) return FASTAR_ERR_ARG;
  if (n_f > FASTAR_MAX_FRAME_KEYS) return FASTAR_ERR_UNSUPPORTED;
  if (F == 0 || n_f == 0 || cache->H == 0) {
    // nothing to merge; the caller's stream still follows the event
    if (codes_ready && cudaStreamWaitEvent(stream, codes_ready, 0) != cudaSuccess) {
      (void)cudaGetLastError();
      return FASTAR_ERR_CUDA;
    }
    return FASTAR_OK;
  }
  if (!k_new || !v_new || !codes_new || !aligned16(k_new) || !aligned16(v_new)) return FASTAR_ERR_ARG;
  if (first_frame < 0 || (int64_t)first_frame + F > 0x7fffff00) return FASTAR_ERR_ARG;
  if (tau != tau) return FASTAR_ERR_ARG;
  const size_t need = merge_ws_bytes(cache->H, n_f, cache->C);
  if (!ws || ws_bytes < need || ((uintptr_t)ws & 255)) return FASTAR_ERR_WORKSPACE;
  return launch_merge(cache, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws,
                      dev_status, stream, codes_ready, rep, planes, search);
}

int fastar_tempcache_merge(const fastar_cache* cache, const void* k_new, const void* v_new,
                           const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                           int32_t* match_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                           cudaStream_t stream) {
  CallRange range("fastar_tempcache_merge");
  return merge_checked(cache, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, ws_bytes,
                       dev_status, stream, nullptr);
}

int fastar_tempcache_merge_ev(const fastar_cache* cache, const void* k_new, const void* v_new,
                              const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                              int32_t* match_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                              cudaStream_t stream, cudaEvent_t codes_ready) {
  CallRange range("fastar_tempcache_merge_ev");
  return merge_checked(cache, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, ws_bytes,
                       dev_status, stream, codes_ready);
}

int fastar_tempcache_merge_rep(const fastar_cache* cache, const void* k_new, const void* v_new,
                               const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                               int rep, const void* planes, int32_t* match_out, void* ws, size_t ws_bytes,
                               int32_t* dev_status, cudaStream_t stream, cudaEvent_t codes_ready) {
  CallRange range("fastar_tempcache_merge_rep");
  return merge_checked(cache, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, ws_bytes,
                       dev_status, stream, codes_ready, rep, planes);
}

int fastar_tempcache_merge_search(const fastar_cache* cache, const void* k_new, const void* v_new,
                                  const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                                  int search, int32_t* match_out, void* ws, size_t ws_bytes,
                                  int32_t* dev_status, cudaStream_t stream, cudaEvent_t codes_ready) {
  CallRange range("fastar_tempcache_merge_search");
  return merge_checked(cache, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, ws_bytes,
                       dev_status, stream, codes_ready, FASTAR_REP_LAST, nullptr, search);
}

int fastar_annca_prune(const uint32_t* q_codes, const uint32_t* p_codes, int H, int F, int n_f,
                       int P, int T, int B, int32_t* kept_idx, int32_t* kept_cnt, void* ws,
                       size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_annca_prune");
  (void)ws;
  (void)ws_bytes;
  if (H < 0 || F < 0 || n_f < 0 || P < 0 || T < 1 || T > 8 || B < 1) return FASTAR_ERR_ARG;
  if (B > 16) return FASTAR_ERR_UNSUPPORTED;
  if (H == 0 || F == 0) return FASTAR_OK;
  if (!kept_cnt || (P > 0 && !kept_idx) || (n_f > 0 && !q_codes) || (P > 0 && !p_codes))
    return FASTAR_ERR_ARG;
  return launch_prune(q_codes, p_codes, H, F, n_f, P, T, B, kept_idx, kept_cnt, dev_status, stream);
}

int fastar_annca_attention(fastar_dtype dt, const void* q, const void* k_p, const void* v_p,
                           const int32_t* kept_idx, const int32_t* kept_cnt, int H, int F, int n_f,
                           int P, int D, float scale, void* out, void* ws, size_t ws_bytes,
                           int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_annca_attention");
  if (!dtype_ok(dt)) return FASTAR_ERR_UNSUPPORTED;
  if (H < 0 || F < 0 || n_f < 0 || P < 0) return FASTAR_ERR_ARG;
  if (!(scale > 0.f && scale < INFINITY)) return FASTAR_ERR_ARG;
  if (!dim_ok(D)) return FASTAR_ERR_UNSUPPORTED;
  if ((size_t)H * F * n_f == 0) return FASTAR_OK;
  if (!q || !out || !kept_cnt || !aligned16(q) || !aligned16(out)) return FASTAR_ERR_ARG;
  if (P > 0 && (!k_p || !v_p || !kept_idx || !aligned16(k_p) || !aligned16(v_p))) return FASTAR_ERR_ARG;
  if (dt == FASTAR_BF16 && D == 128 && P > 0) {
    const size_t need = annca_tc_ws_bytes(H, F, P, D);
    if (!ws || ws_bytes < need || ((uintptr_t)ws & 255)) return FASTAR_ERR_WORKSPACE;
  }
  return launch_annca(dt, q, k_p, v_p, kept_idx, kept_cnt, H, F, n_f, P, D, scale, out, ws, ws_bytes,
                      dev_status, stream);
}

int fastar_annsa_attention(fastar_dtype dt, const void* q, const uint32_t* q_codes,
                           const int32_t* q_perm, const int32_t* q_offsets, int Nq,
                           const fastar_cache* cache, float scale, void* out, float* lse, void* ws,
                           size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_annsa_attention");
  int rc = check_cache(cache);
  if (rc != FASTAR_OK) return rc;
  if (dt != cache->dt) return FASTAR_ERR_ARG;
  if (Nq < 0) return FASTAR_ERR_ARG;
  if (!(scale > 0.f && scale < INFINITY)) return FASTAR_ERR_ARG;
  if (Nq == 0 || cache->H == 0) return FASTAR_OK;
  if (!q || !q_codes || !q_perm || !q_offsets || !out || !aligned16(q) || !aligned16(out))
    return FASTAR_ERR_ARG;
  const size_t need = annsa_ws_bytes(cache->H, Nq, cache->D, cache->T);
  if (need && (!ws || ws_bytes < need || ((uintptr_t)ws & 255))) return FASTAR_ERR_WORKSPACE;
  return launch_annsa(dt, q, q_codes, q_perm, q_offsets, Nq, cache, scale, out, lse, ws,
                      dev_status, stream);
}

int fastar_annsa_attention_part(fastar_dtype dt, const void* q, const uint32_t* q_codes,
                                const int32_t* q_perm, const int32_t* q_offsets, int Nq,
                                const fastar_cache* cache, float scale, int part_base, int part_total,
                                void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_annsa_attention_part");
  (void)q_offsets;
  int rc = check_cache(cache);
  if (rc != FASTAR_OK) return rc;
  if (dt != cache->dt || Nq < 0) return FASTAR_ERR_ARG;
  if (!(scale > 0.f && scale < INFINITY)) return FASTAR_ERR_ARG;
  if (part_total < 1 || part_total > 4 || part_base < 0 || part_base + cache->T > part_total)
    return FASTAR_ERR_ARG;
  if (dt != FASTAR_BF16 || cache->D != 128) return FASTAR_ERR_UNSUPPORTED;
  if (Nq == 0 || cache->H == 0) return FASTAR_OK;
  if (!q || !q_codes || !q_perm || !aligned16(q)) return FASTAR_ERR_ARG;
  const size_t need = annsa_parts_ws_bytes(cache->H, Nq, cache->D, part_total);
  if (!ws || ws_bytes < need || ((uintptr_t)ws & 255)) return FASTAR_ERR_WORKSPACE;
  return launch_annsa_parts(q, q_codes, q_perm, Nq, cache, scale, part_base, part_total, ws, dev_status,
                            stream);
}

int fastar_annsa_combine(int H, int Nq, int D, int part_total, const void* ws, size_t ws_bytes, void* out,
                         float* lse, int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_annsa_combine");
  if (H < 0 || Nq < 0 || part_total < 1 || part_total > 4) return FASTAR_ERR_ARG;
  if (D != 128) return FASTAR_ERR_UNSUPPORTED;
  if (H == 0 || Nq == 0) return FASTAR_OK;
  if (!out || !aligned16(out)) return FASTAR_ERR_ARG;
  const size_t need = annsa_parts_ws_bytes(H, Nq, D, part_total);
  if (!ws || ws_bytes < need || ((uintptr_t)ws & 255)) return FASTAR_ERR_WORKSPACE;
  return launch_annsa_combine(H, Nq, part_total, ws, out, lse, dev_status, stream);
}

}  // extern "C"

static int quant_common(int H, int Nq, int N, int D, float scale, int topk, int bits, const void* q,
                        const void* out, void* ws, size_t ws_bytes) {
  if (H < 0 || Nq < 0 || N < 0 || topk < 0) return FASTAR_ERR_ARG;
  if (!(scale > 0.f && scale < INFINITY)) return FASTAR_ERR_ARG;
  if (bits < 1 || bits > 16) return FASTAR_ERR_UNSUPPORTED;
  if (D != 128) return FASTAR_ERR_UNSUPPORTED;
  if (H == 0 || Nq == 0) return -1;  // nothing to do
  if (!q || !out || !aligned16(q) || !aligned16(out)) return FASTAR_ERR_ARG;
  if (N == 0) return FASTAR_ERR_ARG;
  const size_t need = quant_ws_bytes(H, Nq, N, D, bits);
  if (!ws || ws_bytes < need || ((uintptr_t)ws & 255)) return FASTAR_ERR_WORKSPACE;
  return FASTAR_OK;
}

int fastar_annsa_quant_attention(fastar_dtype dt, const void* q, int Nq, const fastar_cache* cache, float scale,
                                 int topk, int bits, void* out, float* lse, uint32_t* sel_mask, void* ws,
                                 size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_annsa_quant_attention");
  int rc = check_cache(cache);
  if (rc != FASTAR_OK) return rc;
  if (dt != cache->dt) return FASTAR_ERR_ARG;
  if (dt != FASTAR_BF16) return FASTAR_ERR_UNSUPPORTED;
  rc = quant_common(cache->H, Nq, cache->C, cache->D, scale, topk, bits, q, out, ws, ws_bytes);
  if (rc == -1) return FASTAR_OK;
  if (rc != FASTAR_OK) return rc;
  return launch_annsa_quant(q, Nq, cache, scale, topk, bits, out, lse, sel_mask, ws, dev_status, stream);
}

int fastar_annca_quant_attention(fastar_dtype dt, const void* q, const void* k_p, const void* v_p, int H, int Nq,
                                 int P, int D, float scale, int topk, int bits, void* out, uint32_t* sel_mask,
                                 void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  CallRange range("fastar_annca_quant_attention");
  if (!dtype_ok(dt)) return FASTAR_ERR_UNSUPPORTED;
  if (dt != FASTAR_BF16) return FASTAR_ERR_UNSUPPORTED;
  int rc = quant_common(H, Nq, P, D, scale, topk, bits, q, out, ws, ws_bytes);
  if (rc == -1) return FASTAR_OK;
  if (rc != FASTAR_OK) return rc;
  if (!k_p || !v_p || !aligned16(k_p) || !aligned16(v_p)) return FASTAR_ERR_ARG;
  return launch_annca_quant(q, k_p, v_p, H, Nq, P, scale, topk, bits, out, sel_mask, ws, dev_status, stream);
}
