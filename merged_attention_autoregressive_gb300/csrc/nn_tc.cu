// TempCache nearest-neighbour match on the tensor cores (tcgen05, bf16).
//
// For one frame of new keys (FAST-AR summary, paperlayer.ai section 5
// "TempCache": top-1 correspondence; paper.rainbus.top method steps): every
// new key k_j is compared with every candidate group (the groups refreshed in
// the previous frame) by cosine, and matched to the best one (ties: lowest
// slot) iff the cosine reaches tau.
//
// Work units: an item is (head, 128 new keys); a unit is one 128-candidate
// tile of an item (an item without candidates has one empty unit, so that
// its keys' norms are still written).  The kernel is persistent: two CTAs
// per SM, each taking a contiguous range of the units in (head, key tile,
// candidate tile) order, i.e. one or a few items, each over a range of
// candidate tiles.  Several CTAs may share an item; their bests meet in a
// packed 64-bit atomicMax (larger cosine first, then lower slot), so the
// result does not depend on the split.  The CTA is warp-specialised:
//   warp 0     producer: per item, once the MMAs and the norm readers of
//              the previous item are done with it, loads the item's keys (A,
//              128 x 128) by TMA; fills a 2-stage ring of candidate tiles by
//              TMA.  After the first frame of a call the candidates are the
//              rows of the previous frame, contiguous in k_new; for the first
//              frame they are cache rows that an earlier kernel copied, in
//              candidate order, into a contiguous staging buffer.  A head
//              with more first-frame candidates than the staging buffer holds
//              gathers its scattered cache rows with cp.async instead;
//   warp 1     one elected thread issues 8 MMAs (M 128, N 128, K 16) per tile
//              into one of two 128-column fp32 TMEM accumulators; the MMA
//              commit frees the tile's stage, and after an item's last tile
//              the item's A tile;
//   warps 2-9  epilogue: per item the squared norms of the keys (from the A
//              tile), then per tile two warps per TMEM lane quarter, 64
//              columns each in two 32-column passes: a thread scales its
//              key's dot products by the
//              candidates' inverse norms (NaN for a candidate that is not a
//              group or has a zero norm, which drops out of every comparison)
//              and keeps the best (cosine, slot) among the candidates that
//              reach the join threshold (no others can be matched).
// The epilogue reads the candidates' inverse norms and slots from global
// memory (through L1), not from shared memory: while the tensor core streams
// operands out of shared memory, shared-memory loads of other warps wait many
// times longer than L1 loads.
// The kernel also writes the new keys' inverse norms, which the plan of this
// frame masks (NaN for keys that joined another key's group) and which are
// the candidate norms of the next frame.  Barriers, TMEM and, after the first
// frame of a call, the first item's keys and candidate tiles (inputs of the
// call) are set up before the wait on the previous kernel of the stream.
#include <math.h>

#include "common.cuh"
#include "tc.cuh"

namespace fastar {

namespace {

constexpr int kM = 128, kN = 128, kD = 128, kStages = 2, kAcc = 2;
constexpr int kThreads = 320;   // 10 warps
constexpr int kTmemCols = kAcc * kN;

struct NnSmem {
  uint8_t A[kM * kD * 2];
  uint8_t B[kStages][kN * kD * 2];
  float half_best[kM];
  int half_slot[kM];
  uint64_t bar_a;   // the item's A tile has landed (one phase per item)
  uint64_t a_free;  // the item's MMAs and norm readers are done with A
  uint64_t full[kStages], empty[kStages];
  uint64_t tfull[kAcc], tempty[kAcc];
  uint32_t tmem;
};

struct NnArgs {
  const __nv_bfloat16* k_new;  // [H][Nrow][D]
  const __nv_bfloat16* K;      // cache keys [H][C][D]
  int H, n_f, Nrow, fi, C;
  int ldn, ldc;                // row strides of invn_* and cinv (multiples of 4)
  // first frame of a call: candidates = cache slots cand[h][c] (c < ncand[h],
  // stride C), inverse norms cinv[h][c] (NaN: not a usable candidate)
  const int32_t* cand;
  const int32_t* ncand;
  const float* cinv;
  // later frames: candidates = rows of the previous frame; slot prev_slot[h][j]
  // (stride n_f), inverse norm invn_prev[h][j] (NaN for a key that joined
  // another key's group: not a group)
  const int32_t* prev_slot;
  const float* invn_prev;
  float* invn_out;                 // inverse norms of this frame's keys [H][ldn]
  unsigned long long* best_out;    // packed best candidate [H][n_f]
  float tau;                       // join threshold on the cosine
  int from_cache;                  // candidates of every frame are staged cache rows (mean-key groups)
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

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

// The CTA's walk over its units [u, u_end): a segment is one item (h, qt)
// with candidate tiles [ct0, ct1), of which `tiles` hold candidates.  Every
// role walks the same segments.
struct Walk {
  int h = 0, base = 0;  // current head and its first unit
  int ut = 1, nt = 0;   // units and candidate tiles per item of head h
  int nc = 0;           // candidates of head h
};
struct Seg {
  int h, qt, ct0, ct1, tiles, nc;
};

__device__ __forceinline__ bool later_frame(const NnArgs& a) { return a.fi > 0 && !a.from_cache; }
__device__ __forceinline__ int head_cands(const NnArgs& a, int h) {
  return later_frame(a) ? a.n_f : min(max(a.ncand[h], 0), a.C);
}
__device__ __forceinline__ void walk_head(const NnArgs& a, Walk& w, int h) {
  w.h = h;
  w.nc = head_cands(a, h);
  w.nt = (w.nc + kN - 1) / kN;
  w.ut = max(1, w.nt);
}
// The segment that starts at unit u (u inside the walk's current or a later
// head), ending no later than u_end.
__device__ __forceinline__ Seg walk_seg(const NnArgs& a, Walk& w, int atiles, int u, int u_end) {
  while (u >= w.base + atiles * w.ut && w.h + 1 < a.H) {
    w.base += atiles * w.ut;
    walk_head(a, w, w.h + 1);
  }
  const int r = u - w.base;
  Seg s;
  s.h = w.h;
  s.qt = r / w.ut;
  s.ct0 = r % w.ut;
  s.ct1 = min(w.ut, s.ct0 + (u_end - u));
  s.tiles = max(0, min(s.ct1, w.nt) - s.ct0);
  s.nc = w.nc;
  return s;
}
// This CTA's unit range: the total is summed over the heads.
__device__ __forceinline__ void cta_units(const NnArgs& a, int atiles, int& u0, int& u1) {
  long long total = 0;
  for (int h = 0; h < a.H; ++h) {
    const int nc = head_cands(a, h);
    total += (long long)atiles * max(1, (nc + kN - 1) / kN);
  }
  u0 = (int)(total * blockIdx.x / gridDim.x);
  u1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
}

__global__ void __launch_bounds__(kThreads, 2) nn_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                                                           const __grid_constant__ CUtensorMap mapB,
                                                           const __grid_constant__ CUtensorMap mapS,
                                                           NnArgs a, int32_t* st) {
  extern __shared__ uint8_t smem_raw[];
  NnSmem& sm = *reinterpret_cast<NnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int atiles = (a.n_f + kM - 1) / kM;
  const bool later = later_frame(a);
  // After the first frame every head has n_f candidates, so the unit range
  // and the first segment are known before the wait.
  int u0 = 0, u1 = 0, npre = 0;
  if (later) cta_units(a, atiles, u0, u1);
  if (tid == 0) {
    tc::mbar_init(&sm.bar_a, 1);
    tc::mbar_init(&sm.a_free, 9);  // the item's MMA commit and the 8 epilogue warps
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
    tc::prefetch_tensormap(later ? &mapB : &mapS);
    if (later && u0 < u1) {
      Walk w;
      walk_head(a, w, 0);
      const Seg s = walk_seg(a, w, atiles, u0, u1);
      const int row0 = s.h * a.Nrow + a.fi * a.n_f + s.qt * kM;
      tc::mbar_arrive_expect_tx(&sm.bar_a, kM * kD * 2);
      tc::tma_load_2d(sm.A, &mapA, &sm.bar_a, 0, row0);
      tc::tma_load_2d(sm.A + kM * 128, &mapA, &sm.bar_a, 64, row0);
      npre = min(kStages, s.tiles);
      const int rbase = s.h * a.Nrow + (a.fi - 1) * a.n_f;
      for (int t = 0; t < npre; ++t) {
        const int row = rbase + (s.ct0 + t) * kN;
        tc::mbar_arrive_expect_tx(&sm.full[t], kN * kD * 2);
        tc::tma_load_2d(sm.B[t], &mapB, &sm.full[t], 0, row);
        tc::tma_load_2d(sm.B[t] + kN * 128, &mapB, &sm.full[t], 64, row);
      }
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;

  pdl_wait();
  if (block_status_bad(st)) {
    // nothing to do, but the copies issued above land before the CTA leaves
    if (tid == 0 && later && u0 < u1) {
      (void)tc::mbar_wait(&sm.bar_a, 0);
      for (int t = 0; t < npre; ++t) (void)tc::mbar_wait(&sm.full[t], 0);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
    return;
  }
  if (!later) cta_units(a, atiles, u0, u1);
  bool ok = true;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    npre = __shfl_sync(0xffffffffu, npre, 0);
    Walk w;
    walk_head(a, w, 0);
    int g = 0;  // the CTA's tile counter (stage g % kStages)
    int si = 0;
    for (int u = u0; u < u1 && ok; ++si) {
      const Seg s = walk_seg(a, w, atiles, u, u1);
      u += s.ct1 - s.ct0;
      // the item's keys: the first item's were issued before the wait (after
      // the first frame); a later item waits until the previous one is done
      // with the A tile
      if (si > 0 || !later) {
        if (si > 0) ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.a_free, (uint32_t)(si - 1) & 1u));
        if (!ok) break;
        if (lane == 0) {
          const int row0 = s.h * a.Nrow + a.fi * a.n_f + s.qt * kM;
          tc::mbar_arrive_expect_tx(&sm.bar_a, kM * kD * 2);
          tc::tma_load_2d(sm.A, &mapA, &sm.bar_a, 0, row0);
          tc::tma_load_2d(sm.A + kM * 128, &mapA, &sm.bar_a, 64, row0);
        }
      }
      // contiguous candidate rows (k_new of the previous frame, or the
      // staging copy of the first frame's candidates): one TMA per 64-column
      // half of a tile; else a cp.async gather of scattered cache rows
      const bool contiguous = later || s.nc <= a.n_f;
      const CUtensorMap* map = later ? &mapB : &mapS;
      const int rbase = later ? s.h * a.Nrow + (a.fi - 1) * a.n_f : s.h * a.n_f;
      for (int t = 0; t < s.tiles && ok; ++t, ++g) {
        if (si == 0 && t < npre) continue;  // issued before the wait
        const int stg = g % kStages;
        if (g >= kStages)
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.empty[stg], (uint32_t)((g / kStages) - 1) & 1u));
        if (!ok) break;
        if (contiguous) {
          if (lane == 0) {
            const int row = rbase + (s.ct0 + t) * kN;
            tc::mbar_arrive_expect_tx(&sm.full[stg], kN * kD * 2);
            tc::tma_load_2d(sm.B[stg], map, &sm.full[stg], 0, row);
            tc::tma_load_2d(sm.B[stg] + kN * 128, map, &sm.full[stg], 64, row);
          }
        } else {
          const int32_t* srow = a.cand + (size_t)s.h * a.C;
          const int c0 = (s.ct0 + t) * kN;
          const uint32_t tile = tc::smem_u32(sm.B[stg]);
#pragma unroll 4
          for (int i = 0; i < kN * 16 / 32; ++i) {
            const int e = lane + 32 * i, r = e >> 4, ch = e & 15;
            const int c = c0 + r;
            const char* src = nullptr;
            if (c < s.nc) {
              const int sl = __ldg(srow + c);
              if (sl >= 0 && sl < a.C) src = (const char*)(a.K + ((size_t)s.h * a.C + sl) * kD);
            }
            tc::cp_async16(tile + tc::sw128_offset(r, ch, kN), src ? (const void*)(src + ch * 16) : (const void*)a.K,
                           src ? 16u : 0u);
          }
          tc::cp_async_commit();
          asm volatile("cp.async.wait_group 0;" ::: "memory");
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sm.full[stg]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // descriptors are computed on every lane (warp-uniform values) and the
    // elected lane issues
    const uint32_t idesc = tc::idesc_bf16_f32(kM, kN, 0, 0);
    const uint64_t adesc = tc::sdesc_kmajor_sw128(tc::smem_u32(sm.A));
    Walk w;
    walk_head(a, w, 0);
    int g = 0;
    int si = 0;
    for (int u = u0; u < u1 && ok; ++si) {
      const Seg s = walk_seg(a, w, atiles, u, u1);
      u += s.ct1 - s.ct0;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.bar_a, (uint32_t)si & 1u));
      if (!ok) break;
      for (int t = 0; t < s.tiles && ok; ++t, ++g) {
        const int stg = g % kStages, b = g % kAcc;
        ok = tc::mbar_wait(&sm.full[stg], (uint32_t)(g / kStages) & 1u);
        if (ok && g >= kAcc) ok = tc::mbar_wait(&sm.tempty[b], (uint32_t)((g / kAcc) - 1) & 1u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc::tc_fence_after();
        const uint64_t bdesc = tc::sdesc_kmajor_sw128(tc::smem_u32(sm.B[stg]));
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // K step kk: 16 columns (32 bytes) inside 64-column half kk / 4
            const uint32_t off_a = (kk >> 2) * kM * 128 + (kk & 3) * 32;
            const uint32_t off_b = (kk >> 2) * kN * 128 + (kk & 3) * 32;
            tc::mma_bf16(tmem + b * kN, tc::sdesc_add(adesc, off_a), tc::sdesc_add(bdesc, off_b), idesc,
                         kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(&sm.tfull[b]);
          tc::mma_commit(&sm.empty[stg]);
        }
        __syncwarp();
      }
      // the item's MMAs are done with A once this commit arrives
      if (ok && tc::elect_one()) tc::mma_commit(&sm.a_free);
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------- epilogue
    // Every epilogue warp walks all segments (skipping the work once a wait
    // has failed), so that the named barriers below always meet.
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    Walk w;
    walk_head(a, w, 0);
    int g = 0;
    int si = 0;
    for (int u = u0; u < u1; ++si) {
      const Seg s = walk_seg(a, w, atiles, u, u1);
      u += s.ct1 - s.ct0;
      if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.bar_a, (uint32_t)si & 1u));
      const int j = s.qt * kM + row;
      // a warp whose 32 rows are all past the frame's keys (the last key
      // tile of a head) only keeps the accumulator handshake
      const bool rows_live = __any_sync(0xffffffffu, j < a.n_f);
      float na2 = 0.f;
      if (ok && rows_live) na2 = row_sq_norm(sm.A, row, kM);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.a_free);  // this warp is done reading A
      const float ia = na2 > 0.f ? 1.f / sqrtf(na2) : 0.f;
      if (ok && s.ct0 == 0 && half == 0 && j < a.n_f && a.invn_out)
        a.invn_out[(size_t)s.h * a.ldn + j] = na2 > 0.f ? ia : __int_as_float(0x7fc00000);
      // candidate c: inverse norm mrow[c], slot srow[c]
      const float* mrow = later ? a.invn_prev + (size_t)s.h * a.ldn : a.cinv + (size_t)s.h * a.ldc;
      const int32_t* srow = later ? a.prev_slot + (size_t)s.h * a.n_f : a.cand + (size_t)s.h * a.C;
      // Only candidates that can reach tau matter: a key whose best cosine
      // is below tau joins no group, whatever the best candidate.  So the
      // running best starts at the row's threshold, in the units of cs
      // (cosine * |k_j|), lowered by 1e-5 so that rounding cannot drop a
      // candidate the plan's exact test (cosine >= tau) would accept; the
      // plan still decides.  The slot search below then only runs for tiles
      // holding such a candidate.
      float best = na2 > 0.f ? (a.tau - 1e-5f) * sqrtf(na2) : INFINITY;
      // The best candidate's slot: best_slot, or (best_c >= 0) srow[best_c],
      // read only when an exact tie needs it and once at the item's end, so
      // that a new maximum costs no dependent load.
      int best_slot = 0x7fffffff, best_c = -1;
      for (int t = 0; t < s.tiles; ++t, ++g) {
        const int b = g % kAcc;
        const int c0 = (s.ct0 + t) * kN + half * (kN / 2);  // this warp's first column
        // the first pass's candidate inverse norms are loaded before the
        // wait, so that their latency overlaps it (NaN past the last one)
        float mi[32];
        auto load_mi = [&](int c) {
          if (c + 32 <= s.nc) {
            const float4* m4 = reinterpret_cast<const float4*>(mrow + c);  // 16-byte aligned: ld % 4 == 0
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 ib = __ldg(m4 + i);
              mi[4 * i] = ib.x;
              mi[4 * i + 1] = ib.y;
              mi[4 * i + 2] = ib.z;
              mi[4 * i + 3] = ib.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) mi[i] = c + i < s.nc ? __ldg(mrow + c + i) : __int_as_float(0x7fc00000);
          }
        };
        if (rows_live) load_mi(c0);
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.tfull[b], (uint32_t)(g / kAcc) & 1u));
        if (!ok) continue;
        tc::tc_fence_after();
#pragma unroll 1
        for (int part = 0; part < (rows_live ? kN / 64 : 0); ++part) {
          const int c = c0 + part * 32;
          if (c >= s.nc) break;
          if (part > 0) load_mi(c);
          float cs[32];
          tc::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + b * kN + half * (kN / 2) + part * 32, cs);
          // cs = dot * inverse candidate norm, in place (NaN: not a group),
          // two products per instruction (each rounded as on its own)
#pragma unroll
          for (int i = 0; i < 32; i += 2) tc::mul2(cs[i], cs[i + 1], mi[i], mi[i + 1]);
          // phase 1: the largest cosine of the 32 columns (NaN columns are
          // ignored); three-input maxima in four independent chains
          float t4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) t4[c4] = tc::max3(t4[c4], cs[i + c4], cs[i + 4 + c4]);
          }
          const float tmax = tc::max3(t4[0], t4[1], fmaxf(t4[2], t4[3]));
          // phase 2 (only when it can change the answer): the columns
          // attaining it as a bit mask; several equal columns take the
          // lowest slot
          if (tmax >= best) {
            uint32_t e4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int i = 0; i < 32; ++i) e4[i & 3] |= (cs[i] == tmax ? 1u : 0u) << i;
            uint32_t eq = (e4[0] | e4[1]) | (e4[2] | e4[3]);
            if (eq != 0u) {
              if (tmax > best && (eq & (eq - 1u)) == 0u) {
                // one column reaches a new maximum
                best = tmax;
                best_c = c + __ffs(eq) - 1;
              } else {
                // several equal columns, or equal to the current best: the
                // lowest slot wins
                int smin = 0x7fffffff;
                while (eq) {
                  smin = min(smin, __ldg(srow + c + __ffs(eq) - 1));
                  eq &= eq - 1u;
                }
                const int cur = tmax > best ? 0x7fffffff : (best_c >= 0 ? __ldg(srow + best_c) : best_slot);
                best = tmax;
                best_slot = min(smin, cur);
                best_c = -1;
              }
            }
          }
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.tempty[b]);
      }
      if (best_c >= 0) best_slot = __ldg(srow + best_c);
      // merge the two column halves of each row, then publish the item's
      // best (the barrier after the reads keeps the next item's writes out)
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
          atomicMax(a.best_out + (size_t)s.h * a.n_f + j, pack_best(best * ia, best_slot));
      }
      named_bar_sync(1, 256);
    }
  }
  if (!ok) status_set(st, FASTAR_ERR_TIMEOUT);
  if (warp == 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
  pdl_trigger();
}

}  // namespace

int launch_nn_tc(fastar_dtype dt, const void* k_new, int n_f, int Nrow, int H, int fi, const void* K,
                 int C, int D, const int32_t* cand, const int32_t* ncand, const float* cinv, int ldc,
                 const int32_t* prev_slot, const float* invn_prev, float* invn_out, int ldn,
                 unsigned long long* best_out, const void* stage, float tau, int32_t* st, cudaStream_t s,
                 int from_cache) {
  if (dt != FASTAR_BF16 || D != kD) return FASTAR_ERR_UNSUPPORTED;
  if (n_f == 0 || H == 0) return FASTAR_OK;
  if ((ldc & 3) || (ldn & 3) || ldc < C || ldn < n_f) return FASTAR_ERR_ARG;
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
  // Two CTAs per SM (shared memory ~97 KB, TMEM 256 of 512 columns each),
  // but no more CTAs than units (estimated with n_f candidates per head; the
  // kernel counts the first frame's real candidates itself).
  const long long units = (long long)((n_f + kM - 1) / kM) * H * max(1, (n_f + kN - 1) / kN);
  const int grid = (int)std::min<long long>(2LL * sms, units);
  NnArgs a{(const __nv_bfloat16*)k_new, (const __nv_bfloat16*)K, H, n_f, Nrow, fi, C, ldn, ldc, cand, ncand, cinv,
           prev_slot, invn_prev, invn_out, best_out, tau, from_cache};
  fastar::launch_pdl((nn_tc_kernel), dim3(grid), kThreads, smem, s, mapA, mapB, mapS, a, st);
  FASTAR_LAUNCHED(s, "nn_tc");
  return FASTAR_OK;
}

}  // namespace fastar
