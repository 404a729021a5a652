// TempCache: merge the frames of a chunk into the fixed-capacity cache.
//
// FAST-AR summary (paperlayer.ai) section 5 "TempCache" and appendix A,
// Lemma A.1; gist.science technical summary 2.A; paper.rainbus.top method
// steps, TempCache.  For each frame f of the chunk, in order:
//   nn     each new key is matched to the group refreshed in frame f-1 of
//          largest cosine (ties: lowest slot); it joins iff cosine >= tau;
//   plan   one CTA per head groups the matches (lowest index = new
//          representative), ranks the unmatched keys and assigns them free
//          slots, then evicted slots (smallest (last_frame, slot) among the
//          groups not refreshed in frame f); updates size / inserted /
//          evicted and writes the next frame's candidate list;
//   apply  one warp per key writes K, V (count-weighted mean, fp32, rounded
//          to the storage type), m, codes and last_frame.
// The candidates of frame f are exactly the groups that frame f-1 refreshed,
// so each plan writes the candidate list of the next frame; the first frame
// of a call compacts the slots with last_frame == first_frame - 1.
//
// Workspace (caller-owned, no initialisation needed):
//   cand[2][H][C], ncand[2][H], rep_j[H][C], gcnt[H][C],
//   match[H][n_f], plan_slot[H][n_f], plan_kind[H][n_f], plan_cnt[H][n_f],
//   evict[H][n_f],
//   best[H][n_f] (packed best candidate per key, see pack_best),
//   cinv[H][C] (inverse norms of the first frame's candidates),
//   stage[H][n_f][128] bf16 (copies of the first n_f first-frame candidate
//   rows, contiguous, so that the NN kernel can load them by TMA),
//   invn[2][H][n_f] (inverse norms of the keys of the last two frames)
// rep_j/gcnt are indexed by slot; they are clean for every candidate slot
// when a plan starts (only candidates can be matched): cand_init cleans the
// first frame's candidates and each plan the slots it refreshed.  best is
// zeroed when a call starts and again by each plan after it has read it.
#include <math.h>

#include <type_traits>

#include "common.cuh"

namespace fastar {

constexpr int kPlanThreads = 1024;
enum : int { KIND_MEMBER = 0, KIND_LEADER = 1, KIND_INSERT = 2 };

struct MergeWs {
  int32_t* cand[2];
  int32_t* ncand[2];
  int32_t* rep_j;
  int32_t* gcnt;
  int32_t* match;
  int32_t* plan_slot;
  int32_t* plan_kind;
  int32_t* plan_cnt;
  int32_t* evict;
  unsigned long long* best;
  float* cinv;
  float* invn[2];
  __nv_bfloat16* stage;
};

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t merge_ws_bytes(int H, int n_f, int C) {
  size_t b = 0;
  b += 2 * align256((size_t)H * C * 4);   // cand
  b += 2 * align256((size_t)H * 4);       // ncand
  b += 2 * align256((size_t)H * C * 4);   // rep_j, gcnt
  b += 5 * align256((size_t)H * n_f * 4); // match, plan_slot, plan_kind, plan_cnt, evict
  b += align256((size_t)H * n_f * 8);     // best
  b += align256((size_t)H * C * 4);       // cinv
  b += 2 * align256((size_t)H * n_f * 4); // invn
  b += align256((size_t)H * n_f * 128 * 2); // stage
  return b;
}

static MergeWs carve(void* ws, int H, int n_f, int C) {
  char* p = (char*)ws;
  MergeWs w;
  auto take = [&](size_t bytes) { char* r = p; p += align256(bytes); return (int32_t*)r; };
  w.cand[0] = take((size_t)H * C * 4);
  w.cand[1] = take((size_t)H * C * 4);
  w.ncand[0] = take((size_t)H * 4);
  w.ncand[1] = take((size_t)H * 4);
  w.rep_j = take((size_t)H * C * 4);
  w.gcnt = take((size_t)H * C * 4);
  w.match = take((size_t)H * n_f * 4);
  w.plan_slot = take((size_t)H * n_f * 4);
  w.plan_kind = take((size_t)H * n_f * 4);
  w.plan_cnt = take((size_t)H * n_f * 4);
  w.evict = take((size_t)H * n_f * 4);
  w.best = (unsigned long long*)take((size_t)H * n_f * 8);
  w.cinv = (float*)take((size_t)H * C * 4);
  w.invn[0] = (float*)take((size_t)H * n_f * 4);
  w.invn[1] = (float*)take((size_t)H * n_f * 4);
  w.stage = (__nv_bfloat16*)take((size_t)H * n_f * 128 * 2);
  return w;
}

// ---------------------------------------------------------------- cand init
// The slots refreshed in frame prev_frame, in slot order (thread t owns a
// contiguous run of slots, so one load round and one block scan suffice);
// their group accumulators are cleaned for the first plan.
__global__ void __launch_bounds__(kPlanThreads) cand_init_kernel(const int32_t* __restrict__ last_frame,
                                                                 const int32_t* __restrict__ size, int C,
                                                                 int32_t prev_frame, int32_t* cand,
                                                                 int32_t* ncand, unsigned long long* best,
                                                                 int32_t* rep_j, int32_t* gcnt, int n_f,
                                                                 int32_t* st) {
  pdl_wait();
  constexpr int kPer = 16;  // slots per thread and round
  __shared__ int sh[33];
  if (block_status_bad(st)) return;
  const int h = blockIdx.x;
  const int n = min(max(size[h], 0), C);
  const int32_t* lf = last_frame + (size_t)h * C;
  int32_t* out = cand + (size_t)h * C;
  for (int j = threadIdx.x; j < n_f; j += blockDim.x) best[(size_t)h * n_f + j] = 0ull;
  int base = 0;
  for (int r0 = 0; r0 < n; r0 += kPer * kPlanThreads) {
    const int s0 = r0 + threadIdx.x * kPer;
    uint32_t hits = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (s0 + i < n && lf[s0 + i] == prev_frame) hits |= 1u << i;
    int tot;
    int pos = base + block_excl_scan(__popc(hits), sh, &tot);
    while (hits) {
      const int i = __ffs(hits) - 1;
      hits &= hits - 1;
      out[pos++] = s0 + i;
      rep_j[(size_t)h * C + s0 + i] = 0x7fffffff;  // the first plan's group accumulators
      gcnt[(size_t)h * C + s0 + i] = 0;
    }
    base += tot;
  }
  if (threadIdx.x == 0) ncand[h] = base;
  pdl_trigger();
}

// Inverse norms of the first frame's candidates (bf16 rows of 128), one warp
// per candidate, grid-stride over the device-side candidate count; the first
// n_f candidate rows are also copied, in candidate order, into `stage`.
__global__ void __launch_bounds__(256) cand_norm_kernel(const __nv_bfloat16* __restrict__ K, int C,
                                                        const int32_t* __restrict__ cand,
                                                        const int32_t* __restrict__ ncand, float* cinv,
                                                        __nv_bfloat16* stage, int n_f, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  const int h = blockIdx.y, lane = threadIdx.x & 31;
  const int nc = min(max(ncand[h], 0), C);
  for (int c = blockIdx.x * 8 + (threadIdx.x >> 5); c < nc; c += gridDim.x * 8) {
    const int s = cand[(size_t)h * C + c];
    const uint2 u = *reinterpret_cast<const uint2*>(K + ((size_t)h * C + s) * 128 + lane * 4);
    if (c < n_f) *reinterpret_cast<uint2*>(stage + ((size_t)h * n_f + c) * 128 + lane * 4) = u;
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    const float n2 = warp_sum(a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y);
    if (lane == 0) cinv[(size_t)h * C + c] = n2 > 0.f ? 1.f / sqrtf(n2) : __int_as_float(0x7fc00000);
  }
  pdl_trigger();
}

// ---------------------------------------------------------------- NN (SIMT)
template <typename T, int D>
__global__ void __launch_bounds__(256) nn_simt_kernel(const T* __restrict__ k_frame, int n_f, int row_stride_keys,
                                                      const T* __restrict__ K, int C,
                                                      const int32_t* __restrict__ cand,
                                                      const int32_t* __restrict__ ncand,
                                                      unsigned long long* __restrict__ best_out, int32_t* st) {
  pdl_wait();
  constexpr int PER = D / 32;
  if (status_bad(st)) return;
  const int h = blockIdx.y;
  const int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= n_f) return;
  const T* kj = k_frame + ((size_t)h * row_stride_keys + j) * D;
  float kv[PER];
  float nk = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    kv[i] = Elem<T>::ld(kj + lane + 32 * i);
    nk = fmaf(kv[i], kv[i], nk);
  }
  nk = warp_sum(nk);
  const int nc = ncand[h];
  const int32_t* ch = cand + (size_t)h * C;
  float best = -INFINITY;
  int best_slot = 0x7fffffff;
  if (nk > 0.f) {
    const float sk = sqrtf(nk);
    for (int c = 0; c < nc; ++c) {
      const int s = ch[c];
      const T* ks = K + ((size_t)h * C + s) * D;
      float dot = 0.f, nn = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const float v = Elem<T>::ld(ks + lane + 32 * i);
        dot = fmaf(kv[i], v, dot);
        nn = fmaf(v, v, nn);
      }
      dot = warp_sum(dot);
      nn = warp_sum(nn);
      if (nn > 0.f) {
        const float cs = dot / (sk * sqrtf(nn));
        if (cs > best || (cs == best && s < best_slot)) {
          best = cs;
          best_slot = s;
        }
      }
    }
  }
  if (lane == 0) best_out[(size_t)h * n_f + j] = best_slot != 0x7fffffff ? pack_best(best, best_slot) : 0ull;
  pdl_trigger();
}

// ---------------------------------------------------------------- plan
// rep_j / gcnt are clean (INT_MAX / 0) for the candidate slots when a plan
// starts: cand_init cleans the first frame's candidates, and every plan
// cleans the slots its frame refreshed, which are the next frame's
// candidates.  The matches of the frame stay in shared memory.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(int n_f, int C, int32_t f, float tau,
                                                            unsigned long long* __restrict__ best,
                                                            int32_t* __restrict__ match_out, int match_off,
                                                            int match_stride, int32_t* __restrict__ match,
                                                            int32_t* __restrict__ cand_next,
                                                            int32_t* __restrict__ ncand_next,
                                                            int32_t* rep_j, int32_t* gcnt,
                                                            int32_t* __restrict__ plan_slot,
                                                            int32_t* __restrict__ plan_kind,
                                                            int32_t* __restrict__ plan_cnt,
                                                            int32_t* __restrict__ evict,
                                                            const int32_t* __restrict__ last_frame,
                                                            const int32_t* __restrict__ m,
                                                            int32_t* size, int64_t* inserted,
                                                            int64_t* evicted, int32_t* st) {
  pdl_wait();
  extern __shared__ int s_key[];  // [n_f]: matched slot (or -1), later the planned slot
  __shared__ int sh[33];
  __shared__ long long shl[33];
  __shared__ int hist[2048];
  __shared__ int s_lstar, s_nlt, s_found;
  if (block_status_bad(st)) return;
  const int h = blockIdx.x;
  int32_t* rj = rep_j + (size_t)h * C;
  int32_t* gc = gcnt + (size_t)h * C;
  const int32_t* lf = last_frame + (size_t)h * C;
  // 0. the NN decision of every key (best candidate if its cosine reaches
  //    tau), and the groups: count and lowest key index per matched slot
  int unm_local = 0;
  for (int j = threadIdx.x; j < n_f; j += blockDim.x) {
    unsigned long long* bp = best + (size_t)h * n_f + j;
    const unsigned long long key = *bp;
    const int mj = (key != 0ull && best_cos(key) >= tau) ? best_slot(key) : -1;
    s_key[j] = mj;
    match[(size_t)h * n_f + j] = mj;
    if (match_out) match_out[(size_t)h * match_stride + match_off + j] = mj;
    *bp = 0ull;
    if (mj >= 0) {
      atomicMin(&rj[mj], j);
      atomicAdd(&gc[mj], 1);
    } else {
      ++unm_local;
    }
  }
  int U;
  block_excl_scan(unm_local, sh, &U);  // its barriers also order the atomics above
  const int size0 = min(max(size[h], 0), C);
  const int freeslots = C - size0;
  const int n_app = min(freeslots, U);
  const int E = U - n_app;
  // 1. eviction: the E smallest (last_frame, slot) among slots with
  //    last_frame < f that no key of this frame joined
  if (E > 0) {
    // eligible: lf < f, and not a slot matched now (only lf == f-1 can be)
    auto eligible = [&](int s) -> bool {
      const int l = lf[s];
      if (l >= f) return false;
      if (l == f - 1 && gc[s] > 0) return false;
      return true;
    };
    int lo = 0x7fffffff;
    for (int s = threadIdx.x; s < size0; s += blockDim.x)
      if (eligible(s)) lo = min(lo, lf[s]);
    lo = block_min_int(lo, sh);
    if (threadIdx.x == 0) s_found = 0;
    __syncthreads();
    long long below = 0;
    for (long long base = lo; base < (long long)f && lo != 0x7fffffff; base += 2048) {
      for (int i = threadIdx.x; i < 2048; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int s = threadIdx.x; s < size0; s += blockDim.x) {
        if (!eligible(s)) continue;
        const long long d = (long long)lf[s] - base;
        if (d >= 0 && d < 2048) atomicAdd(&hist[(int)d], 1);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        long long cum = below;
        for (int b = 0; b < 2048; ++b) {
          if (cum + hist[b] >= E) {
            s_lstar = (int)(base + b);
            s_nlt = (int)cum;
            s_found = 1;
            break;
          }
          cum += hist[b];
        }
        if (!s_found) s_nlt = (int)cum;
      }
      __syncthreads();
      if (s_found) break;
      below = s_nlt;
      __syncthreads();
    }
    if (!s_found) {
      if (threadIdx.x == 0) status_set(st, FASTAR_ERR_CAPACITY);
      return;
    }
    const int lstar = s_lstar, eq_take = E - s_nlt;
    // ordered selection over slots: chunk of consecutive slots per thread
    const int per = (size0 + blockDim.x - 1) / blockDim.x;
    const int s0 = min(size0, (int)threadIdx.x * per), s1 = min(size0, s0 + per);
    int nlt = 0, neq = 0;
    for (int s = s0; s < s1; ++s) {
      if (!eligible(s)) continue;
      nlt += lf[s] < lstar;
      neq += lf[s] == lstar;
    }
    int tlt, teq;
    int lt_before = block_excl_scan(nlt, sh, &tlt);
    int eq_before = block_excl_scan(neq, sh, &teq);
    int32_t* ev = evict + (size_t)h * n_f;
    for (int s = s0; s < s1; ++s) {
      if (!eligible(s)) continue;
      const int l = lf[s];
      if (l < lstar) {
        ev[lt_before + min(eq_before, eq_take)] = s;
        ++lt_before;
      } else if (l == lstar) {
        if (eq_before < eq_take) ev[lt_before + eq_before] = s;
        ++eq_before;
      }
    }
    __syncthreads();
    // evicted += sum of m over the evicted groups
    long long em = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) em += m[(size_t)h * C + ev[e]];
    em = block_sum_ll(em, shl);
    if (threadIdx.x == 0) evicted[h] += em;
  }
  // 2. per-key plan (ascending j), and the next frame's candidate list; one
  //    block scan counts the unmatched keys (low half) and the candidates
  //    (high half) before each key
  const int32_t* ev = evict + (size_t)h * n_f;
  int urank_base = 0, cand_base = 0;
  for (int j0 = 0; j0 < n_f; j0 += blockDim.x) {
    const int j = j0 + threadIdx.x;
    const bool in = j < n_f;
    const int s = in ? s_key[j] : 0;
    bool leader = false;
    int cnt = 0;
    if (in && s >= 0) {
      leader = rj[s] == j;
      if (leader) cnt = gc[s];
    }
    const int unm = (in && s < 0) ? 1 : 0;
    const int isc = (in && (s < 0 || leader)) ? 1 : 0;
    int tot;
    const int both = block_excl_scan(unm | (isc << 16), sh, &tot);
    const int ur = (both & 0xffff) + urank_base, cp = (both >> 16) + cand_base;
    if (in) {
      const int slot = s >= 0 ? s : (ur < n_app ? size0 + ur : ev[ur - n_app]);
      const int kind = s < 0 ? KIND_INSERT : (leader ? KIND_LEADER : KIND_MEMBER);
      plan_slot[(size_t)h * n_f + j] = slot;
      plan_kind[(size_t)h * n_f + j] = kind;
      plan_cnt[(size_t)h * n_f + j] = cnt;
      if (isc) cand_next[(size_t)h * C + cp] = slot;
      s_key[j] = slot;
    }
    urank_base += tot & 0xffff;
    cand_base += tot >> 16;
  }
  __syncthreads();
  // 3. clean the group accumulators of every slot this frame refreshed
  for (int j = threadIdx.x; j < n_f; j += blockDim.x) {
    const int slot = s_key[j];
    rj[slot] = 0x7fffffff;
    gc[slot] = 0;
  }
  if (threadIdx.x == 0) {
    ncand_next[h] = cand_base;
    size[h] = size0 + n_app;
    inserted[h] += n_f;
  }
  pdl_trigger();
}

// ---------------------------------------------------------------- apply
// One warp per key; lane l handles the D/32 consecutive dimensions starting
// at l * D/32 (one vector access per row).
template <typename T, int D>
__global__ void __launch_bounds__(256) apply_kernel(const T* __restrict__ k_frame, const T* __restrict__ v_frame,
                                                    const uint32_t* __restrict__ codes_frame, int n_f,
                                                    int row_stride_keys, int Tt, int32_t f,
                                                    const int32_t* __restrict__ match,
                                                    const int32_t* __restrict__ plan_slot,
                                                    const int32_t* __restrict__ plan_kind,
                                                    const int32_t* __restrict__ plan_cnt, T* K, T* V,
                                                    int32_t* m, uint32_t* codes, int32_t* last_frame,
                                                    int C, int32_t* st) {
  pdl_wait();
  constexpr int PER = D / 32;
  if (status_bad(st)) return;
  const int h = blockIdx.y;
  const int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= n_f) return;
  const int kind = plan_kind[(size_t)h * n_f + j];
  if (kind == KIND_MEMBER) return;
  const int s = plan_slot[(size_t)h * n_f + j];
  const size_t krow = ((size_t)h * row_stride_keys + j) * D + lane * PER;
  const size_t crow = ((size_t)h * C + s) * D + lane * PER;
  float kv[PER], vv[PER];
  ld_vec<T, PER>(k_frame + krow, kv);
  ld_vec<T, PER>(v_frame + krow, vv);
  int m_new = 1;
  if (kind == KIND_LEADER) {
    const int cnt = plan_cnt[(size_t)h * n_f + j];
    const int m_old = m[(size_t)h * C + s];
    m_new = m_old + cnt;
    float acc[PER];
    ld_vec<T, PER>(V + crow, acc);
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = (float)m_old * acc[i] + vv[i];
    if (cnt > 1) {
      // the other members of the group, in ascending key order
      const int32_t* mt = match + (size_t)h * n_f;
      int left = cnt - 1;
      for (int jj = j + 1; jj < n_f && left > 0; ++jj) {
        if (mt[jj] != s) continue;
        float x[PER];
        ld_vec<T, PER>(v_frame + ((size_t)h * row_stride_keys + jj) * D + lane * PER, x);
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] += x[i];
        --left;
      }
    }
    const float mf = (float)m_new;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = acc[i] / mf;
    st_vec<T, PER>(V + crow, acc);
  } else {
    st_vec<T, PER>(V + crow, vv);
  }
  st_vec<T, PER>(K + crow, kv);
  if (lane == 0) {
    m[(size_t)h * C + s] = m_new;
    last_frame[(size_t)h * C + s] = f;
  }
  for (int t = lane; t < Tt; t += 32)
    codes[((size_t)h * Tt + t) * C + s] = codes_frame[((size_t)h * Tt + t) * row_stride_keys + j];
  pdl_trigger();
}

int launch_nn_tc(fastar_dtype dt, const void* k_new, int n_f, int Nrow, int H, int fi, const void* K,
                 int C, int D, const int32_t* cand, const int32_t* ncand, const float* cinv,
                 const int32_t* prev_slot, const int32_t* prev_kind, const float* invn_prev,
                 float* invn_out, unsigned long long* best_out, const void* stage, float tau, int32_t* st,
                 cudaStream_t s);

template <typename T, int D>
static int merge_impl(const fastar_cache* c, const void* k_new, const void* v_new,
                      const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                      int32_t* match_out, void* ws, int32_t* st, cudaStream_t s) {
  const int H = c->H, C = c->C, Tt = c->T;
  MergeWs w = carve(ws, H, n_f, C);
  // the plan keeps one int per key of a frame in shared memory
  const size_t plan_smem = (size_t)n_f * sizeof(int);
  if (plan_smem > 48 * 1024 &&
      cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan_smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_UNSUPPORTED;
  }
  const int Nrow = F * n_f;
  fastar::launch_pdl((cand_init_kernel), H, kPlanThreads, 0, s, c->last_frame, c->size, C, first_frame - 1,
                                              w.cand[0], w.ncand[0], w.best, w.rep_j, w.gcnt, n_f, st);
  FASTAR_LAUNCHED(s, "cand_init");
  const dim3 wgrid((n_f + 7) / 8, H), wblock(256);
  const bool tc_nn = std::is_same<T, __nv_bfloat16>::value && D == 128;
  if (tc_nn) {
    fastar::launch_pdl((cand_norm_kernel), wgrid, wblock, 0, s, (const __nv_bfloat16*)c->K, C, w.cand[0], w.ncand[0], w.cinv,
                                              w.stage, n_f, st);
    FASTAR_LAUNCHED(s, "cand_norm");
  }
  for (int fi = 0; fi < F; ++fi) {
    const int cur = fi & 1, nxt = cur ^ 1;
    const int32_t f = first_frame + fi;
    const T* kf = (const T*)k_new + (size_t)fi * n_f * D;
    const T* vf = (const T*)v_new + (size_t)fi * n_f * D;
    const uint32_t* cf = codes_new + (size_t)fi * n_f;
    int rc = FASTAR_ERR_UNSUPPORTED;
    if (tc_nn)
      rc = launch_nn_tc(FASTAR_BF16, k_new, n_f, Nrow, H, fi, c->K, C, D, w.cand[cur], w.ncand[cur], w.cinv,
                        w.plan_slot, w.plan_kind, w.invn[(fi + 1) & 1], w.invn[fi & 1], w.best, w.stage,
                        tau, st, s);
    if (rc == FASTAR_ERR_UNSUPPORTED) {
      fastar::launch_pdl((nn_simt_kernel<T, D>), wgrid, wblock, 0, s, kf, n_f, Nrow, (const T*)c->K, C, w.cand[cur],
                                                    w.ncand[cur], w.best, st);
      FASTAR_LAUNCHED(s, "nn_simt");
    } else if (rc != FASTAR_OK) {
      return rc;
    }
    fastar::launch_pdl((plan_kernel), H, kPlanThreads, (size_t)n_f * sizeof(int), s, 
        n_f, C, f, tau, w.best, match_out, fi * n_f, Nrow, w.match, w.cand[nxt], w.ncand[nxt], w.rep_j,
        w.gcnt, w.plan_slot, w.plan_kind, w.plan_cnt, w.evict, c->last_frame, c->m, c->size, c->inserted,
        c->evicted, st);
    FASTAR_LAUNCHED(s, "plan");
    fastar::launch_pdl((apply_kernel<T, D>), wgrid, wblock, 0, s, kf, vf, cf, n_f, Nrow, Tt, f, w.match, w.plan_slot,
                                                w.plan_kind, w.plan_cnt, (T*)c->K, (T*)c->V, c->m,
                                                c->codes, c->last_frame, C, st);
    FASTAR_LAUNCHED(s, "apply");
  }
  return launch_csr(c->codes, H * Tt, C, c->size, Tt, 1 << c->B, c->perm, c->offsets, st, s);
}

int launch_merge(const fastar_cache* c, const void* k_new, const void* v_new,
                 const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                 int32_t* match_out, void* ws, int32_t* st, cudaStream_t s) {
  if (c->dt == FASTAR_F32 && c->D == 64)
    return merge_impl<float, 64>(c, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, st, s);
  if (c->dt == FASTAR_F32 && c->D == 128)
    return merge_impl<float, 128>(c, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, st, s);
  if (c->dt == FASTAR_BF16 && c->D == 64)
    return merge_impl<__nv_bfloat16, 64>(c, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, st, s);
  if (c->dt == FASTAR_BF16 && c->D == 128)
    return merge_impl<__nv_bfloat16, 128>(c, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, st, s);
  return FASTAR_ERR_UNSUPPORTED;
}

}  // namespace fastar
