// TempCache: merge the frames of a chunk into the fixed-capacity cache.
//
// FAST-AR summary (paperlayer.ai) section 5 "TempCache" and appendix A,
// Lemma A.1; gist.science technical summary 2.A; paper.rainbus.top method
// steps, TempCache.  For each frame f of the chunk, in order:
//   nn     each new key is matched to the group refreshed in frame f-1 of
//          largest cosine (ties: lowest slot); it joins iff cosine >= tau;
//   plan   one CTA per head groups the matches in shared memory (lowest
//          index = new representative), ranks the unmatched keys and assigns them free
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
//   cand[2][H][C], ncand[2][H],
//   match[H][n_f], plan_slot[H][n_f], plan_kind[H][n_f], plan_cnt[H][n_f],
//   evict[H][n_f],
//   best[H][n_f] (packed best candidate per key, see pack_best),
//   cinv[H][ldc] (inverse norms of the first frame's candidates; NaN for an
//   unusable one; ldc = C rounded up to 4),
//   stage[H][n_f][128] bf16 (copies of the first n_f first-frame candidate
//   rows, contiguous, so that the NN kernel can load them by TMA),
//   invn[2][H][ldn] (inverse norms of the keys of the last two frames; the
//   plan of a frame sets NaN for its keys that joined another key's group,
//   which are no candidates of the next frame; ldn = n_f rounded up to 4)
// best is zeroed when a call starts and again by each plan after it has
// read it.
#include <math.h>

#include <type_traits>

#include "common.cuh"

namespace fastar {

constexpr int kPlanThreads = 1024;
enum : int { KIND_MEMBER = 0, KIND_LEADER = 1, KIND_INSERT = 2 };

struct MergeWs {
  int32_t* cand[2];
  int32_t* ncand[2];
  int32_t* match;
  int32_t* plan_slot;
  int32_t* plan_kind;
  int32_t* plan_cnt;
  int32_t* evict;
  unsigned long long* best;
  float* cinv;
  float* invn[2];
  __nv_bfloat16* stage;
  void* qsmall;  // the quantised search's per-dimension ranges
  int ldc, ldn;  // row strides of cinv and invn (multiples of 4 floats)
};

size_t quant_nn_ws_bytes(int H, int n_f);
int launch_quant_nn(const void* k_frame, long long a_rows, int n_f, int H, const void* K, int C, const int32_t* cand,
                    const int32_t* ncand, int bits, void* ws_small, void* codes, float* dec_inv, int ld_inv,
                    unsigned long long* best, int32_t* st, cudaStream_t s);

static inline int round4(int x) { return (x + 3) & ~3; }

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t merge_ws_bytes(int H, int n_f, int C) {
  size_t b = 0;
  b += 2 * align256((size_t)H * C * 4);   // cand
  b += 2 * align256((size_t)H * 4);       // ncand
  b += 5 * align256((size_t)H * n_f * 4); // match, plan_slot, plan_kind, plan_cnt, evict
  b += align256((size_t)H * n_f * 8);     // best
  b += align256((size_t)H * round4(C) * 4);       // cinv
  b += 2 * align256((size_t)H * round4(n_f) * 4); // invn
  b += align256((size_t)H * n_f * 128 * 2); // stage (the quantised search's codes)
  b += align256(quant_nn_ws_bytes(H, n_f)); // quantised search ranges
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
  w.match = take((size_t)H * n_f * 4);
  w.plan_slot = take((size_t)H * n_f * 4);
  w.plan_kind = take((size_t)H * n_f * 4);
  w.plan_cnt = take((size_t)H * n_f * 4);
  w.evict = take((size_t)H * n_f * 4);
  w.best = (unsigned long long*)take((size_t)H * n_f * 8);
  w.ldc = round4(C);
  w.ldn = round4(n_f);
  w.cinv = (float*)take((size_t)H * w.ldc * 4);
  w.invn[0] = (float*)take((size_t)H * w.ldn * 4);
  w.invn[1] = (float*)take((size_t)H * w.ldn * 4);
  w.stage = (__nv_bfloat16*)take((size_t)H * n_f * 128 * 2);
  w.qsmall = (void*)take(quant_nn_ws_bytes(H, n_f));
  return w;
}

// ---------------------------------------------------------------- cand init
// The slots refreshed in frame prev_frame, in slot order (thread t owns a
// contiguous run of slots, so one load round and one block scan suffice).
__global__ void __launch_bounds__(kPlanThreads) cand_init_kernel(const int32_t* __restrict__ last_frame,
                                                                 const int32_t* __restrict__ size, int C,
                                                                 int32_t prev_frame, int32_t* cand,
                                                                 int32_t* ncand, unsigned long long* best,
                                                                 int n_f,
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
    }
    base += tot;
  }
  if (threadIdx.x == 0) ncand[h] = base;
  pdl_trigger();
}

// Inverse norms of the first frame's candidates (bf16 rows of 128): a warp
// handles kNormCands consecutive candidates (all rows loaded first), over a
// grid-stride range of the device-side candidate count; the first n_f
// candidate rows are also copied, in candidate order, into `stage`.
constexpr int kNormCands = 4;
__global__ void __launch_bounds__(256) cand_norm_kernel(const __nv_bfloat16* __restrict__ K, int C,
                                                        const int32_t* __restrict__ cand,
                                                        const int32_t* __restrict__ ncand, float* cinv,
                                                        int ldc, __nv_bfloat16* stage, int n_f, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  const int h = blockIdx.y, lane = threadIdx.x & 31;
  const int nc = min(max(ncand[h], 0), C);
  const int step = gridDim.x * 8 * kNormCands;
  for (int c0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * kNormCands; c0 < nc; c0 += step) {
    int sl[kNormCands];
#pragma unroll
    for (int u = 0; u < kNormCands; ++u) sl[u] = c0 + u < nc ? cand[(size_t)h * C + c0 + u] : -1;
    uint2 row[kNormCands];
#pragma unroll
    for (int u = 0; u < kNormCands; ++u)
      if (sl[u] >= 0) row[u] = *reinterpret_cast<const uint2*>(K + ((size_t)h * C + sl[u]) * 128 + lane * 4);
#pragma unroll
    for (int u = 0; u < kNormCands; ++u) {
      const int c = c0 + u;
      if (sl[u] < 0) {
        if (c < nc && lane == 0) cinv[(size_t)h * ldc + c] = __int_as_float(0x7fc00000);
        continue;
      }
      if (c < n_f) *reinterpret_cast<uint2*>(stage + ((size_t)h * n_f + c) * 128 + lane * 4) = row[u];
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&row[u].x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&row[u].y));
      const float n2 = warp_sum(a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y);
      if (lane == 0) cinv[(size_t)h * ldc + c] = n2 > 0.f ? 1.f / sqrtf(n2) : __int_as_float(0x7fc00000);
    }
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

// ---------------------------------------------------------------- NN over every earlier frame
// The search variant that looks for the nearest earlier group over every
// previous frame through the LSH buckets (gist.science technical summary
// 2.A: the nearest earlier key is found with LSH or quantisation; the
// method's default searches the previous frame only): the candidates of new
// key j are the live groups sharing an LSH bucket with it in some table,
// read from the cache's bucket CSR (rebuilt before every frame); a group
// found through table t is skipped when an earlier table already offered
// it.  One warp per key, one candidate per lane (32 at a time): each lane
// reads its candidate's slot, its earlier-table codes and its whole row
// (independent loads), and the key is read from shared memory; the warp
// keeps the top-1 cosine, ties to the lowest slot, packed as by the NN
// kernels; the plan merges iff the cosine reaches tau.
template <typename T, int D>
__global__ void __launch_bounds__(256) nn_lsh_kernel(const T* __restrict__ k_frame, int n_f, int row_stride_keys,
                                                     const uint32_t* __restrict__ codes_frame,
                                                     const T* __restrict__ K, const uint32_t* __restrict__ codes,
                                                     const int32_t* __restrict__ size,
                                                     const int32_t* __restrict__ perm,
                                                     const int32_t* __restrict__ offsets, int C, int Tt, int nb,
                                                     unsigned long long* __restrict__ best_out, int32_t* st) {
  pdl_wait();
  constexpr int PER = D / 32;
  constexpr int VN = 16 / (int)sizeof(T);  // elements per 16-byte load
  __shared__ float s_key[8][D];
  if (status_bad(st)) return;
  const int h = blockIdx.y, wib = threadIdx.x >> 5;
  const int j = blockIdx.x * 8 + wib;
  const int lane = threadIdx.x & 31;
  if (j >= n_f) return;  // a whole warp; no block barrier follows
  const T* kj = k_frame + ((size_t)h * row_stride_keys + j) * D;
  float nk = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const float v = Elem<T>::ld(kj + lane + 32 * i);
    s_key[wib][lane + 32 * i] = v;
    nk = fmaf(v, v, nk);
  }
  nk = warp_sum(nk);
  __syncwarp();
  uint32_t kc[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) kc[t] = t < Tt ? codes_frame[((size_t)h * Tt + t) * row_stride_keys + j] : 0u;
  const int n_live = min(max(size[h], 0), C);
  float best = -INFINITY;
  int best_slot = 0x7fffffff;
  bool bad = false;
  if (nk > 0.f) {
    const float sk = sqrtf(nk);
    for (int t = 0; t < Tt; ++t) {
      if (kc[t] >= (uint32_t)nb) {
        bad = true;
        continue;
      }
      const int32_t* off = offsets + ((size_t)h * Tt + t) * (nb + 1);
      const int a = min(max(off[kc[t]], 0), n_live);
      const int b = min(max(off[kc[t] + 1], a), n_live);
      const int32_t* pt = perm + ((size_t)h * Tt + t) * C;
      for (int p0 = a; p0 < b; p0 += 32) {
        const int p = p0 + lane;
        if (p >= b) continue;
        const int s = pt[p];
        if (s < 0 || s >= n_live) {
          bad = true;
          continue;
        }
        bool seen = false;
        for (int u = 0; u < t; ++u) seen |= codes[((size_t)h * Tt + u) * C + s] == kc[u];
        if (seen) continue;
        const T* ks = K + ((size_t)h * C + s) * D;
        float dot = 0.f, nn = 0.f;
#pragma unroll 4
        for (int d = 0; d < D; d += VN) {
          float kv[VN];
          ld_vec<T, VN>(ks + d, kv);
#pragma unroll
          for (int e = 0; e < VN; ++e) {
            dot = fmaf(s_key[wib][d + e], kv[e], dot);
            nn = fmaf(kv[e], kv[e], nn);
          }
        }
        if (nn > 0.f) {
          const float cs = dot / (sk * sqrtf(nn));
          if (cs > best || (cs == best && s < best_slot)) {
            best = cs;
            best_slot = s;
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int os = __shfl_xor_sync(0xffffffffu, best_slot, o);
    if (ob > best || (ob == best && os < best_slot)) {
      best = ob;
      best_slot = os;
    }
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    best_out[(size_t)h * n_f + j] = best_slot != 0x7fffffff ? pack_best(best, best_slot) : 0ull;
    if (bad) status_set(st, FASTAR_ERR_DEVICE_ARG);
  }
  pdl_trigger();
}

// ---------------------------------------------------------------- plan
// The frame's matches and groups live in shared memory: s_key[n_f] holds
// each key's matched slot (later its planned slot), and an open-addressing
// hash table of 2^lg_tab entries (at least 4/3 of n_f, so it never fills)
// maps each matched slot to its group: lowest key index and count.
__device__ __forceinline__ int plan_hash(int slot, int lg_tab) {
  return (int)(((uint32_t)slot * 2654435761u) >> (32 - lg_tab));
}
// Entry of `slot`, inserting it when absent.
__device__ __forceinline__ int plan_insert(int* tab_slot, int slot, int lg_tab) {
  const int mask = (1 << lg_tab) - 1;
  int e = plan_hash(slot, lg_tab);
  for (int i = 0; i <= mask; ++i) {
    const int prev = atomicCAS(&tab_slot[e], -1, slot);
    if (prev == -1 || prev == slot) return e;
    e = (e + 1) & mask;
  }
  return -1;  // cannot happen: the table has more entries than keys
}
// Entry of `slot`, or -1 when no key of the frame matched it.
__device__ __forceinline__ int plan_find(const int* tab_slot, int slot, int lg_tab) {
  const int mask = (1 << lg_tab) - 1;
  int e = plan_hash(slot, lg_tab);
  for (int i = 0; i <= mask; ++i) {
    const int v = tab_slot[e];
    if (v == slot) return e;
    if (v == -1) return -1;
    e = (e + 1) & mask;
  }
  return -1;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(int n_f, int C, int32_t f, float tau, int lg_tab,
                                                            unsigned long long* __restrict__ best,
                                                            int32_t* __restrict__ match_out, int match_off,
                                                            int match_stride, int32_t* __restrict__ match,
                                                            int32_t* __restrict__ cand_next,
                                                            int32_t* __restrict__ ncand_next,
                                                            int32_t* __restrict__ plan_slot,
                                                            int32_t* __restrict__ plan_kind,
                                                            int32_t* __restrict__ plan_cnt,
                                                            int32_t* __restrict__ evict,
                                                            const int32_t* __restrict__ last_frame,
                                                            const int32_t* __restrict__ m,
                                                            int32_t* size, int64_t* inserted,
                                                            int64_t* evicted, float* __restrict__ invn, int ldn,
                                                            int any_frame, int32_t* st) {
  pdl_wait();
  extern __shared__ int plan_smem[];
  const int ntab = 1 << lg_tab;
  int* s_key = plan_smem;              // [n_f]
  int* tab_slot = s_key + n_f;         // [ntab], -1 = empty
  int* tab_min = tab_slot + ntab;      // [ntab] lowest key index of the group
  int* tab_cnt = tab_min + ntab;       // [ntab] keys in the group
  __shared__ int sh[33];
  __shared__ long long shl[33];
  __shared__ int hist[2048];
  __shared__ int s_lstar, s_nlt, s_found;
  if (block_status_bad(st)) return;
  const int h = blockIdx.x;
  const int32_t* lf = last_frame + (size_t)h * C;
  for (int e = threadIdx.x; e < ntab; e += blockDim.x) {
    tab_slot[e] = -1;
    tab_min[e] = 0x7fffffff;
    tab_cnt[e] = 0;
  }
  __syncthreads();
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
      const int e = plan_insert(tab_slot, mj, lg_tab);
      atomicMin(&tab_min[e], j);
      atomicAdd(&tab_cnt[e], 1);
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
    // eligible: lf < f, and not a slot matched now (only lf == f-1 can be,
    // unless the search covers every earlier frame)
    auto eligible = [&](int s) -> bool {
      const int l = lf[s];
      if (l >= f) return false;
      if ((any_frame || l == f - 1) && plan_find(tab_slot, s, lg_tab) >= 0) return false;
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
      const int e = plan_find(tab_slot, s, lg_tab);
      leader = tab_min[e] == j;
      if (leader) cnt = tab_cnt[e];
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
      // a key that joined another key's group is no candidate of the next
      // frame: the tensor-core NN reads this as "not a group"
      if (invn && kind == KIND_MEMBER) invn[(size_t)h * ldn + j] = __int_as_float(0x7fc00000);
      if (isc) cand_next[(size_t)h * C + cp] = slot;
    }
    urank_base += tot & 0xffff;
    cand_base += tot >> 16;
  }
  if (threadIdx.x == 0) {
    ncand_next[h] = cand_base;
    size[h] = size0 + n_app;
    inserted[h] += n_f;
  }
  pdl_trigger();
}

// ---------------------------------------------------------------- apply
// One warp per kApplyKeys consecutive keys (their plan records, then all of
// their rows, are loaded before any is used); lane l handles the D/32
// consecutive dimensions starting at l * D/32 (one vector access per row).
// With the mean-key representative (planes != nullptr; FAST-AR summary,
// paperlayer.ai, appendix C) a joined group's key becomes the count-weighted
// mean of its keys, summed like the value, and its codes the hash of the
// stored mean: one warp-reduced dot product per hyperplane, a zero
// projection giving bit 0.
constexpr int kApplyKeys = 4;
// Three CTAs per SM: the register budget of four spills the rows in flight,
// that of two halves the warps hiding the dependent loads (14B-like frame:
// 57 us at three, 59 at four, 75 at two; eight keys per warp at two, 71).

// Sign bits of 16 warp-wide dot products: p[r] is this lane's share of
// product r.  A reduce-scatter over the warp (lanes exchange half of their
// values at each of four steps) leaves lane l with the sum over 16 lanes of
// product (l >> 1) & 15, one more exchange completes it over all 32 lanes,
// and a ballot over the even lanes collects the 16 signs (bit r = [sum_r > 0]).
__device__ __forceinline__ uint32_t warp_sign_bits16(float (&p)[16], int lane) {
  float a[8], b4[4], c2[2];
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float keep = h16 ? p[i + 8] : p[i], send = h16 ? p[i] : p[i + 8];
    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = h8 ? a[i + 4] : a[i], send = h8 ? a[i] : a[i + 4];
    b4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = h4 ? b4[i + 2] : b4[i], send = h4 ? b4[i] : b4[i + 2];
    c2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const float keep = h2 ? c2[1] : c2[0], send = h2 ? c2[0] : c2[1];
  float sum = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  const uint32_t even = __ballot_sync(0xffffffffu, sum > 0.f) & 0x55555555u;
  // lane 2r holds product r: compact the even bits
  uint32_t bits = 0u;
#pragma unroll
  for (int r = 0; r < 16; ++r) bits |= ((even >> (2 * r)) & 1u) << r;
  return bits;
}

template <typename T>
__device__ __forceinline__ float stored(float x) {
  T y;
  Elem<T>::st(&y, x);
  return Elem<T>::ld(&y);
}
template <typename T, int D, bool kMean>
__global__ void __launch_bounds__(256, 3) apply_kernel(const T* __restrict__ k_frame, const T* __restrict__ v_frame,
                                                    const uint32_t* __restrict__ codes_frame, int n_f,
                                                    int row_stride_keys, int Tt, int32_t f,
                                                    const int32_t* __restrict__ match,
                                                    const int32_t* __restrict__ plan_slot,
                                                    const int32_t* __restrict__ plan_kind,
                                                    const int32_t* __restrict__ plan_cnt, T* K, T* V,
                                                    int32_t* m, uint32_t* codes, int32_t* last_frame,
                                                    int C, const T* __restrict__ planes, int Bb,
                                                    int32_t* st) {
  constexpr int PER = D / 32;
  const int h = blockIdx.y;
  const int j0 = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kApplyKeys;
  const int lane = threadIdx.x & 31;
  // the keys' k and v rows are inputs of the call (an earlier kernel of the
  // call has already waited for their producers): load them before the wait
  using Raw = typename VecOf<T, PER>::type;
  Raw kv[kApplyKeys], vv[kApplyKeys], vo[kApplyKeys], ko[kApplyKeys];
#pragma unroll
  for (int u = 0; u < kApplyKeys; ++u) {
    if (j0 + u >= n_f) continue;
    const size_t krow = ((size_t)h * row_stride_keys + j0 + u) * D + lane * PER;
    kv[u] = ld_raw<T, PER>(k_frame + krow);
    vv[u] = ld_raw<T, PER>(v_frame + krow);
  }
  pdl_wait();
  if (status_bad(st)) return;
  int kind[kApplyKeys], slot[kApplyKeys], cnt[kApplyKeys], m_old[kApplyKeys];
#pragma unroll
  for (int u = 0; u < kApplyKeys; ++u) {
    const int j = j0 + u;
    kind[u] = KIND_MEMBER;
    slot[u] = 0;
    cnt[u] = 0;
    if (j < n_f) {
      kind[u] = plan_kind[(size_t)h * n_f + j];
      slot[u] = plan_slot[(size_t)h * n_f + j];
      cnt[u] = plan_cnt[(size_t)h * n_f + j];
    }
  }
#pragma unroll
  for (int u = 0; u < kApplyKeys; ++u) {
    m_old[u] = 0;
    if (kind[u] == KIND_LEADER) {
      m_old[u] = m[(size_t)h * C + slot[u]];
      vo[u] = ld_raw<T, PER>(V + ((size_t)h * C + slot[u]) * D + lane * PER);
      if constexpr (kMean) ko[u] = ld_raw<T, PER>(K + ((size_t)h * C + slot[u]) * D + lane * PER);
    }
  }
#pragma unroll
  for (int u = 0; u < kApplyKeys; ++u) {
    if (kind[u] == KIND_MEMBER) continue;
    const int j = j0 + u, s = slot[u];
    const size_t crow = ((size_t)h * C + s) * D + lane * PER;
    int m_new = 1;
    if (kind[u] == KIND_LEADER) {
      m_new = m_old[u] + cnt[u];
      float acc[PER], x[PER], kacc[PER];
      raw_to_float<T, PER>(vo[u], acc);
      raw_to_float<T, PER>(vv[u], x);
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = (float)m_old[u] * acc[i] + x[i];
      if constexpr (kMean) {
        raw_to_float<T, PER>(ko[u], kacc);
        raw_to_float<T, PER>(kv[u], x);
#pragma unroll
        for (int i = 0; i < PER; ++i) kacc[i] = (float)m_old[u] * kacc[i] + x[i];
      }
      if (cnt[u] > 1) {
        // the other members of the group, in ascending key order: the warp
        // tests 32 keys per step and adds the members it finds in order
        const int32_t* mt = match + (size_t)h * n_f;
        int left = cnt[u] - 1;
        for (int base = j + 1; base < n_f && left > 0; base += 32) {
          const int jj = base + lane;
          unsigned bits = __ballot_sync(0xffffffffu, jj < n_f && mt[jj] == s);
          while (bits != 0u && left > 0) {
            const int k = __ffs(bits) - 1;
            bits &= bits - 1u;
            ld_vec<T, PER>(v_frame + ((size_t)h * row_stride_keys + base + k) * D + lane * PER, x);
#pragma unroll
            for (int i = 0; i < PER; ++i) acc[i] += x[i];
            if constexpr (kMean) {
              ld_vec<T, PER>(k_frame + ((size_t)h * row_stride_keys + base + k) * D + lane * PER, x);
#pragma unroll
              for (int i = 0; i < PER; ++i) kacc[i] += x[i];
            }
            --left;
          }
        }
      }
      const float mf = (float)m_new;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = acc[i] / mf;
      st_vec<T, PER>(V + crow, acc);
      if constexpr (kMean) {
#pragma unroll
        for (int i = 0; i < PER; ++i) kacc[i] = kacc[i] / mf;
        st_vec<T, PER>(K + crow, kacc);
        // codes of the stored (rounded) mean key
#pragma unroll
        for (int i = 0; i < PER; ++i) kacc[i] = stored<T>(kacc[i]);
        // one bit per hyperplane, 16 hyperplanes per warp reduction
        const int R = Tt * Bb;  // <= 64
        uint64_t signs = 0ull;
        for (int r0 = 0; r0 < R; r0 += 16) {
          float p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            p[i] = 0.f;
            if (r0 + i < R) {
              float pr[PER];
              ld_vec<T, PER>(planes + (size_t)(r0 + i) * D + lane * PER, pr);
#pragma unroll
              for (int e = 0; e < PER; ++e) p[i] = fmaf(pr[e], kacc[e], p[i]);
            }
          }
          signs |= (uint64_t)warp_sign_bits16(p, lane) << r0;
        }
        if (lane < Tt)
          codes[((size_t)h * Tt + lane) * C + s] = (uint32_t)(signs >> (lane * Bb)) & ((1u << Bb) - 1u);
      }
    } else {
      st_raw<T, PER>(V + crow, vv[u]);
    }
    // K and codes of key j (a mean-key group's were written above)
    const bool own_key = !kMean || kind[u] != KIND_LEADER;
    if (own_key) st_raw<T, PER>(K + crow, kv[u]);
    if (lane == 0) {
      m[(size_t)h * C + s] = m_new;
      last_frame[(size_t)h * C + s] = f;
    }
    if (own_key)
      for (int t = lane; t < Tt; t += 32)
        codes[((size_t)h * Tt + t) * C + s] = codes_frame[((size_t)h * Tt + t) * row_stride_keys + j];
  }
  pdl_trigger();
}

int launch_nn_tc(fastar_dtype dt, const void* k_new, int n_f, int Nrow, int H, int fi, const void* K,
                 int C, int D, const int32_t* cand, const int32_t* ncand, const float* cinv, int ldc,
                 const int32_t* prev_slot, const float* invn_prev, float* invn_out, int ldn,
                 unsigned long long* best_out, const void* stage, float tau, int32_t* st, cudaStream_t s,
                 int from_cache);

template <typename T, int D>
static int merge_impl(const fastar_cache* c, const void* k_new, const void* v_new,
                      const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                      int32_t* match_out, void* ws, int32_t* st, cudaStream_t s, cudaEvent_t codes_ready,
                      int rep, const void* planes, int search) {
  const int H = c->H, C = c->C, Tt = c->T;
  // search over every earlier frame (LSH candidates): the cache CSR is
  // rebuilt before each frame and a warp per key walks its buckets
  const bool lsh = search == FASTAR_SEARCH_LSH;
  // quantised search (TempCache-Quant): the previous frame's groups, ranked
  // by approximate cosine to their b-bit codes, the best merged iff its
  // exact cosine reaches tau
  const bool quant = (search & 0xff) == FASTAR_SEARCH_QUANT;
  const int qbits = search >> 8;
  if ((lsh || quant) && rep != FASTAR_REP_LAST) return FASTAR_ERR_UNSUPPORTED;
  if (quant && (!std::is_same<T, __nv_bfloat16>::value || D != 128 || qbits < 1 || qbits > 16))
    return FASTAR_ERR_UNSUPPORTED;
  // mean-key groups: every frame's candidates are cache rows (their stored
  // means), staged like the first frame's; the apply re-hashes merged keys
  const bool mean_key = rep == FASTAR_REP_MEAN;
  MergeWs w = carve(ws, H, n_f, C);
  // the plan keeps one int per key of a frame and a hash table of the
  // frame's groups (3 ints per entry, at least 4/3 n_f entries) in shared
  // memory
  int lg_tab = 6;
  while ((1 << lg_tab) * 3 < n_f * 4) ++lg_tab;
  const size_t plan_smem = (size_t)n_f * sizeof(int) + 3 * ((size_t)sizeof(int) << lg_tab);
  if (plan_smem > 48 * 1024 &&
      cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan_smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_UNSUPPORTED;
  }
  const int Nrow = F * n_f;
  const dim3 wgrid((n_f + 7) / 8, H), wblock(256);
  const bool tc_nn = !lsh && !quant && std::is_same<T, __nv_bfloat16>::value && D == 128;
  if (lsh) {
    // every frame's search reads its keys' codes
    if (codes_ready && cudaStreamWaitEvent(s, codes_ready, 0) != cudaSuccess) {
      (void)cudaGetLastError();
      return FASTAR_ERR_CUDA;
    }
    codes_ready = nullptr;
  } else {
    fastar::launch_pdl((cand_init_kernel), H, kPlanThreads, 0, s, c->last_frame, c->size, C, first_frame - 1,
                       w.cand[0], w.ncand[0], w.best, n_f, st);
    FASTAR_LAUNCHED(s, "cand_init");
  }
  if (tc_nn) {
    fastar::launch_pdl((cand_norm_kernel), dim3((n_f + 8 * kNormCands - 1) / (8 * kNormCands), H), wblock, 0, s, (const __nv_bfloat16*)c->K, C, w.cand[0], w.ncand[0], w.cinv,
                                              w.ldc, w.stage, n_f, st);
    FASTAR_LAUNCHED(s, "cand_norm");
  }
  for (int fi = 0; fi < F; ++fi) {
    const int cur = fi & 1, nxt = cur ^ 1;
    const int32_t f = first_frame + fi;
    const T* kf = (const T*)k_new + (size_t)fi * n_f * D;
    const T* vf = (const T*)v_new + (size_t)fi * n_f * D;
    const uint32_t* cf = codes_new + (size_t)fi * n_f;
    int rc = FASTAR_ERR_UNSUPPORTED;
    if (lsh) {
      rc = launch_csr(c->codes, H * Tt, C, c->size, Tt, 1 << c->B, c->perm, c->offsets, st, s);
      if (rc != FASTAR_OK) return rc;
      fastar::launch_pdl((nn_lsh_kernel<T, D>), wgrid, wblock, 0, s, kf, n_f, Nrow, cf, (const T*)c->K,
                         (const uint32_t*)c->codes, c->size, c->perm, c->offsets, C, Tt, 1 << c->B, w.best, st);
      FASTAR_LAUNCHED(s, "nn_lsh");
    }
    if (quant) {
      rc = launch_quant_nn((const void*)kf, Nrow, n_f, H, c->K, C, w.cand[cur],
                           w.ncand[cur], qbits, w.qsmall, w.stage, w.cinv, w.ldc, w.best, st, s);
      if (rc != FASTAR_OK) return rc;
    }
    if (tc_nn && mean_key && fi > 0) {
      // the candidates the previous plan listed, with the keys its apply wrote
      fastar::launch_pdl((cand_norm_kernel), dim3((n_f + 8 * kNormCands - 1) / (8 * kNormCands), H), wblock, 0, s,
                         (const __nv_bfloat16*)c->K, C, w.cand[cur], w.ncand[cur], w.cinv, w.ldc, w.stage, n_f, st);
      FASTAR_LAUNCHED(s, "cand_norm");
    }
    if (tc_nn)
      rc = launch_nn_tc(FASTAR_BF16, k_new, n_f, Nrow, H, fi, c->K, C, D, w.cand[cur], w.ncand[cur], w.cinv,
                        w.ldc, w.plan_slot, w.invn[(fi + 1) & 1], w.invn[fi & 1], w.ldn, w.best, w.stage,
                        tau, st, s, mean_key ? 1 : 0);
    if (rc == FASTAR_ERR_UNSUPPORTED && !lsh && !quant) {
      fastar::launch_pdl((nn_simt_kernel<T, D>), wgrid, wblock, 0, s, kf, n_f, Nrow, (const T*)c->K, C, w.cand[cur],
                                                    w.ncand[cur], w.best, st);
      FASTAR_LAUNCHED(s, "nn_simt");
    } else if (rc != FASTAR_OK) {
      return rc;
    }
    fastar::launch_pdl((plan_kernel), H, kPlanThreads, plan_smem, s, n_f, C, f, tau, lg_tab, w.best, match_out,
                       fi * n_f, Nrow, w.match, w.cand[nxt], w.ncand[nxt], w.plan_slot, w.plan_kind, w.plan_cnt,
                       w.evict, c->last_frame, c->m, c->size, c->inserted, c->evicted,
                       tc_nn ? w.invn[fi & 1] : nullptr, w.ldn, lsh ? 1 : 0, st);
    FASTAR_LAUNCHED(s, "plan");
    // the first kernel that reads codes_new (or v_new): wait for them here
    if (fi == 0 && codes_ready && cudaStreamWaitEvent(s, codes_ready, 0) != cudaSuccess) {
      (void)cudaGetLastError();
      return FASTAR_ERR_CUDA;
    }
    const dim3 agrid((n_f + 8 * kApplyKeys - 1) / (8 * kApplyKeys), H);
    if (mean_key)
      fastar::launch_pdl((apply_kernel<T, D, true>), agrid, wblock, 0, s, kf, vf, cf, n_f, Nrow, Tt, f, w.match,
                         w.plan_slot, w.plan_kind, w.plan_cnt, (T*)c->K, (T*)c->V, c->m, c->codes, c->last_frame,
                         C, (const T*)planes, c->B, st);
    else
      fastar::launch_pdl((apply_kernel<T, D, false>), agrid, wblock, 0, s, kf, vf, cf, n_f, Nrow, Tt, f, w.match,
                         w.plan_slot, w.plan_kind, w.plan_cnt, (T*)c->K, (T*)c->V, c->m, c->codes, c->last_frame,
                         C, (const T*)nullptr, c->B, st);
    FASTAR_LAUNCHED(s, "apply");
  }
  return launch_csr(c->codes, H * Tt, C, c->size, Tt, 1 << c->B, c->perm, c->offsets, st, s);
}

int launch_merge(const fastar_cache* c, const void* k_new, const void* v_new,
                 const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                 int32_t* match_out, void* ws, int32_t* st, cudaStream_t s, cudaEvent_t codes_ready,
                 int rep, const void* planes, int search) {
#define FASTAR_MERGE(T, D)                                                                                   \
  return merge_impl<T, D>(c, k_new, v_new, codes_new, F, n_f, first_frame, tau, match_out, ws, st, s, codes_ready, \
                          rep, planes, search)
  if (c->dt == FASTAR_F32 && c->D == 64) FASTAR_MERGE(float, 64);
  if (c->dt == FASTAR_F32 && c->D == 128) FASTAR_MERGE(float, 128);
  if (c->dt == FASTAR_BF16 && c->D == 64) FASTAR_MERGE(__nv_bfloat16, 64);
  if (c->dt == FASTAR_BF16 && c->D == 128) FASTAR_MERGE(__nv_bfloat16, 128);
#undef FASTAR_MERGE
  return FASTAR_ERR_UNSUPPORTED;
}

}  // namespace fastar
