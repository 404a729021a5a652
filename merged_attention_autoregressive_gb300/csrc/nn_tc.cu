// TempCache nearest-neighbour match on the tensor cores (tcgen05, bf16).
//
// For one frame of new keys (FAST-AR summary, paperlayer.ai section 5
// "TempCache": top-1 correspondence; paper.rainbus.top method steps): every
// new key k_j is compared with every candidate group (the groups refreshed in
// the previous frame) by cosine, and matched to the best one (ties: lowest
// slot) iff the cosine reaches tau.
//
// One CTA owns 128 new keys of one head and one slice of the candidates (the
// candidates are split over gridDim.y CTAs; the split minimises the launch's
// rounds of SM slots times the CTA cost).  The new keys arrive by TMA (two
// 64-column boxes, 128-byte swizzle).  The slots and inverse norms of the
// CTA's candidates are staged in shared memory once, by the epilogue warps
// while the first tiles load.  The CTA is warp-specialised:
//   warp 0     producer: fills a 4-stage ring of 64-row candidate tiles by
//              TMA.  After the first frame of a call the candidates are the
//              rows of the previous frame, contiguous in k_new; for the first
//              frame they are cache rows that an earlier kernel copied, in
//              candidate order, into a contiguous staging buffer.  A head
//              with more first-frame candidates than the staging buffer holds
//              gathers its scattered cache rows with cp.async instead;
//   warp 1     one thread issues 8 MMAs (M 128, N 64, K 16) per tile into one
//              of four 64-column fp32 TMEM accumulators; the MMA commit frees
//              the tile's stage;
//   warps 2-9  epilogue: two warps per TMEM lane quarter, 32 columns each;
//              a thread scales its key's dot products by the candidates'
//              inverse norms (NaN for a candidate with a zero norm, which
//              drops out of every comparison) and keeps the best
//              (cosine, slot) among the candidates that are groups and
//              reach the join threshold (no others can be matched).
// At the end the two halves of a row are merged and the CTA's best of each
// key is folded into a packed 64-bit word with atomicMax (larger cosine
// first, then lower slot), so the result does not depend on CTA order.  The
// epilogue also writes the new keys' inverse norms, which are the candidate
// norms of the next frame.
#include <math.h>

#include "common.cuh"
#include "tc.cuh"

namespace fastar {

namespace {

constexpr int kM = 128, kN = 64, kD = 128, kStages = 4, kAcc = 4;
constexpr int kThreads = 320;  // 10 warps
constexpr int kMember = 0;     // plan kind of a key that joined a group it does not represent
constexpr int kMetaCap = 1408; // candidates whose slot / inverse norm are staged per CTA

struct NnSmem {
  uint8_t A[kM * kD * 2];
  uint8_t B[kStages][kN * kD * 2];
  int mslot[kMetaCap];
  float minv[kMetaCap];
  float half_best[kM];
  int half_slot[kM];
  uint64_t bar_a;
  uint64_t full[kStages], empty[kStages];
  uint64_t tfull[kAcc], tempty[kAcc];
  uint32_t tmem;
};

__device__ __forceinline__ float row_sq_norm(const uint8_t* tile, int r, int rows) {
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint4 u = *(const uint4*)(tile + tc::sw128_offset(r, c, rows));
    const __nv_bfloat162* p = (const __nv_bfloat162*)&u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(p[k]);
      s = fmaf(f.x, f.x, s);
      s = fmaf(f.y, f.y, s);
    }
  }
  return s;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

struct NnArgs {
  const __nv_bfloat16* k_new;  // [H][Nrow][D]
  const __nv_bfloat16* K;      // cache keys [H][C][D]
  int n_f, Nrow, fi, C;
  // first frame of a call: candidates = cache slots cand[h][c] (c < ncand[h]),
  // inverse norms cinv[h][c] (stride C)
  const int32_t* cand;
  const int32_t* ncand;
  const float* cinv;
  // later frames: candidates = rows of the previous frame, a group iff its
  // plan kind is not "member"; inverse norms invn_prev[h][j] (stride n_f)
  const int32_t* prev_slot;
  const int32_t* prev_kind;
  const float* invn_prev;
  float* invn_out;                 // inverse norms of this frame's keys [H][n_f]
  unsigned long long* best_out;    // packed best candidate [H][n_f]
  float tau;                       // join threshold on the cosine
};

__device__ __forceinline__ void cand_meta(const NnArgs& a, int h, int c, int& slot, float& inv) {
  if (a.fi == 0) {
    slot = a.cand[(size_t)h * a.C + c];
    inv = a.cinv[(size_t)h * a.C + c];
  } else {
    slot = a.prev_kind[(size_t)h * a.n_f + c] != kMember ? a.prev_slot[(size_t)h * a.n_f + c] : -1;
    inv = a.invn_prev[(size_t)h * a.n_f + c];
  }
}

__global__ void __launch_bounds__(kThreads, 2) nn_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                                                           const __grid_constant__ CUtensorMap mapB,
                                                           const __grid_constant__ CUtensorMap mapS,
                                                           NnArgs a, int32_t* st) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  NnSmem& sm = *reinterpret_cast<NnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  if (block_status_bad(st)) return;
  const int h = blockIdx.z, m0 = blockIdx.x * kM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nc = (a.fi == 0) ? min(max(a.ncand[h], 0), a.C) : a.n_f;
  const int ttot = (nc + kN - 1) / kN;
  const int tb0 = (int)((long long)ttot * blockIdx.y / gridDim.y);
  const int tb1 = (int)((long long)ttot * (blockIdx.y + 1) / gridDim.y);
  const int ntiles = tb1 - tb0;
  const int cbase = tb0 * kN, cend = min(nc, tb1 * kN);

  if (tid == 0) {
    tc::mbar_init(&sm.bar_a, 1);
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&sm.full[s], 1);   // producer lane 0 (with the TMA bytes, or after the gather)
      tc::mbar_init(&sm.empty[s], 1);  // MMA commit
    }
    for (int b = 0; b < kAcc; ++b) {
      tc::mbar_init(&sm.tfull[b], 1);   // MMA commit
      tc::mbar_init(&sm.tempty[b], 8);  // 8 epilogue warps
    }
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&mapA);
    tc::prefetch_tensormap(&mapB);
    if (a.fi == 0) tc::prefetch_tensormap(&mapS);
    const int row0 = h * a.Nrow + a.fi * a.n_f + m0;
    tc::mbar_arrive_expect_tx(&sm.bar_a, kM * kD * 2);
    tc::tma_load_2d(sm.A, &mapA, &sm.bar_a, 0, row0);
    tc::tma_load_2d(sm.A + kM * 128, &mapA, &sm.bar_a, 64, row0);
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem, kAcc * kN);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // The epilogue warps stage the candidates' slots and inverse norms while
  // the producer and the MMA issuer already start on the first tiles; named
  // barrier 2 (epilogue + producer) publishes them.  The producer needs the
  // slots only when it gathers scattered cache rows, otherwise it just
  // arrives.
  if (warp >= 2) {
    for (int c = cbase + tid - 64; c < cbase + ntiles * kN && c - cbase < kMetaCap; c += kThreads - 64) {
      int sl = -1;
      float inv = __int_as_float(0x7fc00000);
      if (c < cend) cand_meta(a, h, c, sl, inv);
      sm.mslot[c - cbase] = sl;
      sm.minv[c - cbase] = sl >= 0 ? inv : __int_as_float(0x7fc00000);
    }
    named_bar_sync(2, kThreads - 32);
  } else if (warp == 0) {
    if (a.fi > 0 || nc <= a.n_f) named_bar_arrive(2, kThreads - 32);
    else named_bar_sync(2, kThreads - 32);
  }
  const uint32_t tmem = sm.tmem;
  bool ok = true;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (a.fi > 0 || nc <= a.n_f) {
      // contiguous candidate rows (k_new of the previous frame, or the
      // staging copy of the first frame's candidates): one TMA per 64-column
      // half of a tile
      const CUtensorMap* map = a.fi > 0 ? &mapB : &mapS;
      const int rbase = a.fi > 0 ? h * a.Nrow + (a.fi - 1) * a.n_f : h * a.n_f;
      if (lane == 0) {
        for (int t = 0; t < ntiles && ok; ++t) {
          const int s = t % kStages;
          if (t >= kStages) ok = tc::mbar_wait(&sm.empty[s], (uint32_t)((t / kStages) - 1) & 1u);
          if (!ok) break;
          const int row = rbase + (tb0 + t) * kN;
          tc::mbar_arrive_expect_tx(&sm.full[s], kN * kD * 2);
          tc::tma_load_2d(sm.B[s], map, &sm.full[s], 0, row);
          tc::tma_load_2d(sm.B[s] + kN * 128, map, &sm.full[s], 64, row);
        }
      }
    } else {
      // scattered cache rows: cp.async gather, a stage is released once its
      // copies have landed (kStages - 1 tiles later in the issue order)
      for (int t = 0; t < ntiles + kStages - 1; ++t) {
        if (t < ntiles) {
          const int s = t % kStages;
          if (t >= kStages) ok = ok && tc::mbar_wait(&sm.empty[s], (uint32_t)((t / kStages) - 1) & 1u);
          const int c0 = (tb0 + t) * kN;
          const uint32_t tile = tc::smem_u32(sm.B[s]);
#pragma unroll 4
          for (int i = 0; i < kN * 16 / 32; ++i) {
            const int e = lane + 32 * i, r = e >> 4, ch = e & 15;
            const int c = c0 + r;
            const char* src = nullptr;
            if (c < nc) {
              int sl = -1;
              if (c - cbase < kMetaCap) {
                sl = sm.mslot[c - cbase];
              } else {
                float unused;
                cand_meta(a, h, c, sl, unused);
              }
              if (sl >= 0) src = (const char*)(a.K + ((size_t)h * a.C + sl) * kD);
            }
            tc::cp_async16(tile + tc::sw128_offset(r, ch, kN), src ? (const void*)(src + ch * 16) : (const void*)a.K,
                           src ? 16u : 0u);
          }
        }
        tc::cp_async_commit();  // one group per iteration (empty past the last tile)
        if (t >= kStages - 1) {
          asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sm.full[(t - (kStages - 1)) % kStages]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t idesc = tc::idesc_bf16_f32(kM, kN, 0, 0);
    if (ntiles > 0) ok = tc::mbar_wait(&sm.bar_a, 0);
    for (int t = 0; t < ntiles && ok; ++t) {
      const int s = t % kStages, b = t % kAcc;
      ok = tc::mbar_wait(&sm.full[s], (uint32_t)(t / kStages) & 1u);
      if (ok && t >= kAcc) ok = tc::mbar_wait(&sm.tempty[b], (uint32_t)((t / kAcc) - 1) & 1u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc::tc_fence_after();
      if (lane == 0) {
        const uint32_t a0 = tc::smem_u32(sm.A), b0 = tc::smem_u32(sm.B[s]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off_a = (kk >> 2) * kM * 128 + (kk & 3) * 32;
          const uint32_t off_b = (kk >> 2) * kN * 128 + (kk & 3) * 32;
          tc::mma_bf16(tmem + b * kN, tc::sdesc_kmajor_sw128(a0 + off_a), tc::sdesc_kmajor_sw128(b0 + off_b),
                       idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sm.tfull[b]);
        tc::mma_commit(&sm.empty[s]);
      }
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.bar_a, 0));
    const float na2 = row_sq_norm(sm.A, row, kM);
    const float ia = na2 > 0.f ? 1.f / sqrtf(na2) : 0.f;
    const int j = m0 + row;
    if (half == 0 && blockIdx.y == 0 && j < a.n_f && a.invn_out)
      a.invn_out[(size_t)h * a.n_f + j] = na2 > 0.f ? ia : __int_as_float(0x7fc00000);
    // Only candidates that can reach tau matter: a key whose best cosine is
    // below tau joins no group, whatever the best candidate.  So the running
    // best starts at the row's threshold, in the units of cs (cosine * |k_j|),
    // lowered by 1e-5 so that rounding cannot drop a candidate the plan's
    // exact test (cosine >= tau) would accept; the plan still decides.  The
    // slot search below then only runs for tiles holding such a candidate.
    float best = na2 > 0.f ? (a.tau - 1e-5f) * sqrtf(na2) : INFINITY;
    int best_slot = 0x7fffffff;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int b = t % kAcc;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.tfull[b], (uint32_t)(t / kAcc) & 1u));
      if (!ok) break;
      tc::tc_fence_after();
      const int c0 = (tb0 + t) * kN;
      const int nval = min(kN, nc - c0);
      const int col0 = half * 32;
      if (col0 < nval) {
        float v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + b * kN + col0, v);
        const int m_off = c0 + col0 - cbase;  // index of column col0 in the staged metadata
        // cs = dot * inverse candidate norm, in place (NaN: not a group)
        float* cs = v;
        if (m_off + 32 <= kMetaCap) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 ib = *reinterpret_cast<const float4*>(&sm.minv[m_off + i]);
            cs[i] *= ib.x;
            cs[i + 1] *= ib.y;
            cs[i + 2] *= ib.z;
            cs[i + 3] *= ib.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            int sl = -1;
            float ib = __int_as_float(0x7fc00000);
            if (col0 + i < nval) cand_meta(a, h, c0 + col0 + i, sl, ib);
            cs[i] = sl >= 0 ? cs[i] * ib : __int_as_float(0x7fc00000);
          }
        }
        // phase 1: the tile's largest cosine (NaN columns are ignored); four
        // independent chains keep the dependency depth short
        float t4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 32; ++i) t4[i & 3] = fmaxf(t4[i & 3], cs[i]);
        const float tmax = fmaxf(fmaxf(t4[0], t4[1]), fmaxf(t4[2], t4[3]));
        // phase 2 (only when it can change the answer): the columns attaining
        // it as a bit mask; several equal columns take the lowest slot
        if (tmax >= best) {
          uint32_t e4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int i = 0; i < 32; ++i) e4[i & 3] |= (cs[i] == tmax ? 1u : 0u) << i;
          uint32_t eq = (e4[0] | e4[1]) | (e4[2] | e4[3]);
          auto slot_at = [&](int i) -> int {
            if (m_off + i < kMetaCap) return sm.mslot[m_off + i];
            int sl;
            float unused;
            cand_meta(a, h, c0 + col0 + i, sl, unused);
            return sl;
          };
          int smin = 0x7fffffff;
          const bool any = eq != 0u;
          while (eq) {
            smin = min(smin, slot_at(__ffs(eq) - 1));
            eq &= eq - 1u;
          }
          if (any && (tmax > best || smin < best_slot)) {
            best = tmax;
            best_slot = smin;
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.tempty[b]);
    }
    // merge the two column halves of each row (epilogue warps only)
    if (half == 1) {
      sm.half_best[row] = best;
      sm.half_slot[row] = best_slot;
    }
    named_bar_sync(1, 256);
    if (half == 0) {
      const float b2 = sm.half_best[row];
      const int s2 = sm.half_slot[row];
      if (b2 > best || (b2 == best && s2 < best_slot)) {
        best = b2;
        best_slot = s2;
      }
      if (ok && j < a.n_f && na2 > 0.f && best_slot != 0x7fffffff)
        atomicMax(a.best_out + (size_t)h * a.n_f + j, pack_best(best * ia, best_slot));
    }
  }
  if (!ok) status_set(st, FASTAR_ERR_TIMEOUT);
  if (warp == 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kAcc * kN);
  pdl_trigger();
}

}  // namespace

int launch_nn_tc(fastar_dtype dt, const void* k_new, int n_f, int Nrow, int H, int fi, const void* K,
                 int C, int D, const int32_t* cand, const int32_t* ncand, const float* cinv,
                 const int32_t* prev_slot, const int32_t* prev_kind, const float* invn_prev,
                 float* invn_out, unsigned long long* best_out, const void* stage, float tau, int32_t* st,
                 cudaStream_t s) {
  if (dt != FASTAR_BF16 || D != kD) return FASTAR_ERR_UNSUPPORTED;
  if (n_f == 0 || H == 0) return FASTAR_OK;
  CUtensorMap mapA, mapB, mapS;
  if (make_tmap_bf16_2d(&mapA, k_new, (uint64_t)H * Nrow, kD, kM, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  if (make_tmap_bf16_2d(&mapB, k_new, (uint64_t)H * Nrow, kD, kN, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  if (make_tmap_bf16_2d(&mapS, stage, (uint64_t)H * n_f, kD, kN, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  const size_t smem = sizeof(NnSmem) + 1024;
  if (cudaFuncSetAttribute(nn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_CUDA;
  }
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  (void)cudaGetLastError();
  // split the candidates over gridDim.y CTAs (the expected candidate count is
  // n_f: the groups the previous frame refreshed)
  const int atiles = (n_f + kM - 1) / kM;
  const int btiles = (n_f + kN - 1) / kN;
  // Two CTAs fit an SM.  A CTA costs a fixed start (A tile, metadata,
  // TMEM; about kStartTiles tile times) plus its tiles, and the launch takes
  // as many rounds as the CTAs need SM slots: pick the split with the least
  // rounds x CTA cost among those whose metadata fits the staging area.
  constexpr int kStartTiles = 6;
  const int min_split = max(1, (btiles * kN + kMetaCap - 1) / kMetaCap);
  const long long slots = 2LL * sms;
  int split = min_split;
  long long best_cost = -1;
  for (int sp = min_split; sp <= min(16, btiles); ++sp) {
    const long long rounds = ((long long)atiles * H * sp + slots - 1) / slots;
    const long long cost = rounds * (kStartTiles + (btiles + sp - 1) / sp);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      split = sp;
    }
  }
  split = max(1, min(split, btiles));
  NnArgs a{(const __nv_bfloat16*)k_new, (const __nv_bfloat16*)K, n_f, Nrow, fi, C, cand, ncand, cinv,
           prev_slot, prev_kind, invn_prev, invn_out, best_out, tau};
  fastar::launch_pdl((nn_tc_kernel), dim3(atiles, split, H), kThreads, smem, s, mapA, mapB, mapS, a, st);
  FASTAR_LAUNCHED(s, "nn_tc");
  return FASTAR_OK;
}

}  // namespace fastar
