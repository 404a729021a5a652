// AnnCA and AnnSA attention on the tensor cores (tcgen05 + TMEM, bf16).
//
// One CTA owns 128 queries (one per softmax thread) and walks their keys 64
// at a time through a warp-specialised pipeline:
//   warp 0     producer: AnnCA's queries (one TMA box pair), then the key
//              rows and, separately, the value rows and mask metadata of
//              every tile (AnnCA: TMA tile loads of the compacted kept rows,
//              or of the prompt's own rows where a frame keeps all of them;
//              AnnSA: TMA tile::gather4 loads, four slot rows each, into the
//              128-byte swizzled layout, or two 64-row boxes for a run of
//              consecutive slots in one-bucket descriptions; 2-stage rings),
//              each as soon as its stage is free: a key stage once its QK
//              product is done, a value stage once its PV product is; row
//              sources and metadata are fetched one tile ahead;
//   warp 1     MMA issuer: S_j = Q K_j^T (M 128, N 64, K 128) into one of two
//              TMEM buffers and O += P_j V_j (M 128, N 128, K 64; P_j read
//              from TMEM, V as an MN-major operand) into the TMEM
//              accumulator, each as soon as its inputs are ready (QK at most
//              one tile ahead of PV);
//   warps 2-5  softmax, one thread per query row (AnnSA: each also gathers
//              its query row): read S_j from TMEM, apply the scale, the
//              + ln m bias and the mask, keep a running max and sum in base 2,
//              write P_j (bf16 pairs) over S_j in TMEM.  The running max is
//              only raised (and O in TMEM rescaled) when a tile's maximum
//              exceeds it by more than 2^8, so P stays <= 256 and rescaling
//              is rare.
// At the end the softmax threads read O from TMEM, stage their rows in shared
// memory and write them out one row per warp instruction.
//
// AnnCA (gist.science technical summary 2.B): the CTA owns 128 queries of
// one frame and walks the frame's kept prompt tokens; it writes the
// normalised output.
// AnnSA (gist.science 2.C; paper.rainbus.top method steps; + ln m from
// paperlayer.ai appendix A, Lemma A.1): one launch covers every LSH table
// t (grid y).  The CTA owns 128 consecutive queries of the chunk in the
// bucket order of table t (the query CSR) and walks the cache slots of the
// buckets they span (the cache CSR, sorted by code too).  A slot is allowed
// for a query iff their table-t codes agree and no earlier table already
// allowed it, so every allowed pair is visited exactly once over the T
// tables.  The slots of a query's own table-t bucket form one run of the
// CTA's key list (from the cache CSR offsets); a warp skips every 32-key
// chunk that no run of its queries meets.  With one table the CTA writes the
// normalised output and the log-sum-exp; with more, each table writes its
// partial (normalised by its own sum, in fp16, with its running max and sum)
// and a combine kernel merges the T partials of each query.
#include <cuda_fp16.h>
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "tc.cuh"

namespace fastar {

namespace {

constexpr int kM = 128, kN = 64, kD = 128, kMaxT = 4, kStages = 2;
constexpr int kThreads = 192;  // producer, MMA issuer, 4 softmax warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.f;  // raise the running max only when exceeded by more than this (log2)
constexpr uint32_t kIdlePolls = 1u << 22;  // MMA issuer: bound on polls that find nothing ready

struct AttnSmem {
  uint8_t Q[kM * kD * 2];
  uint8_t K[kStages][kN * kD * 2];
  uint8_t V[kStages][kN * kD * 2];
  float bias[kStages][kN];                      // AnnSA: log2 m of the tile's slots
  uint32_t kcodes[kStages][kMaxT - 1][kN];      // AnnSA: slot codes of the tables before t
  uint64_t bar_q;
  uint64_t kfull[kStages], vfull[kStages], kempty[kStages], vempty[kStages];
  uint64_t sfull[2], pready[2], odone, fin;
  uint32_t tmem;
};
// At the end the output rows are staged through Q and K (free by then):
// 16 KB per softmax warp.
static_assert(sizeof(((AttnSmem*)0)->Q) + sizeof(((AttnSmem*)0)->K) >= 4 * 32 * kD * 4, "staging space");

struct CaArgs {
  const __nv_bfloat16* k_p;
  const __nv_bfloat16* v_p;
  const int32_t* kept_idx;
  const int32_t* kept_cnt;
  int F, n_f, P, P64;  // P64: rows per (head, frame) of the compacted kept K / V
  __nv_bfloat16* out;
};

struct SaArgs {
  const __nv_bfloat16* q;
  const uint32_t* q_codes;
  const int32_t* q_perm;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const int32_t* m;
  const uint32_t* codes;
  const int32_t* size;
  const int32_t* perm;
  const int32_t* offsets;
  int C, T, nb;
  __half* ws_o;  // [T][H][Nq][D] per-table partials, normalised by their own sums (fp16)
  float2* ws_ml; // [T][H][Nq] their (max in log2 units, sum)
  __nv_bfloat16* out;
  float* lse;
  int slot0;       // first partial slot of this call (table t writes slot0 + t)
  int parts_only;  // write partials even for one table (no output)
  // optional per-query selection (the quantised matcher): key position p of
  // query i is allowed only if bit p % 32 of row_mask[(h Nq + i) mask_words
  // + p / 32] is set (with the one-bucket description, position = slot)
  const uint32_t* row_mask;
  int mask_words;
};

// Wait until the PV product of key tile j has landed in O (and, since one
// thread issues every MMA in order, all products before it); called by a
// softmax thread that has seen S_{j+1}.  The commit after PV_j arrives on
// vempty[j % kStages].  A parity wait is only sound while the barrier is at
// most one phase behind the awaited one: the previous phase on that barrier
// (PV_{j-2}) has completed, because QK_{j+1}, which the caller has seen
// complete, was issued after PV_{j-1} (QK runs at most one tile ahead of PV) and the MMAs complete in issue order; and the next phase
// (PV_{j+2}) cannot complete before the caller has written P_{j+2}.
__device__ __forceinline__ bool wait_pv(AttnSmem& sm, int j) {
  return tc::mbar_wait(&sm.vempty[j % kStages], (uint32_t)(j / kStages) & 1u);
}

// 2^x by the SFU instruction (relative error about 2^-22; results below
// 2^-126 flush to 0, and 2^-inf is 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bits c (0..63) of the key tile with lo <= c < hi.
__device__ __forceinline__ uint64_t range_bits(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 64);
  if (hi <= lo) return 0ull;
  const uint64_t below_hi = hi >= 64 ? ~0ull : ((1ull << hi) - 1ull);
  const uint64_t below_lo = (1ull << lo) - 1ull;
  return below_hi & ~below_lo;
}

// AnnCA: the kept prompt rows of each (head, frame), compacted in kept
// order into Kc/Vc [(h * F + f) * P64 + k][D] (P64 = P rounded up to 64),
// with zero rows up to the next multiple of 64, so that the attention kernel
// loads whole key tiles with two TMA boxes.  One CTA per 64-row tile, a
// warp per row at a time (8 bytes per lane).  A (head, frame) that keeps
// every token is not copied: the attention kernel reads the prompt's rows.
__global__ void __launch_bounds__(256) annca_compact_kernel(const __nv_bfloat16* __restrict__ k_p,
                                                            const __nv_bfloat16* __restrict__ v_p,
                                                            const int32_t* __restrict__ kept_idx,
                                                            const int32_t* __restrict__ kept_cnt, int F, int P,
                                                            int P64, __nv_bfloat16* __restrict__ kc,
                                                            __nv_bfloat16* __restrict__ vc, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  const int t = blockIdx.x, f = blockIdx.y, h = blockIdx.z;
  const int cnt = min(max(kept_cnt[(size_t)h * F + f], 0), P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // a (head, frame) that keeps every prompt token reads the prompt's own
  // rows (the kept list is the prompt in order): nothing to copy
  if (cnt < P && t * kN < cnt) {
    bool bad = false;
    for (int r = warp; r < kN; r += 8) {
      const int k = t * kN + r;
      const size_t dst = (((size_t)h * F + f) * P64 + k) * kD + lane * 4;
      uint2 ku = make_uint2(0u, 0u), vu = make_uint2(0u, 0u);
      if (k < cnt) {
        const int p = kept_idx[((size_t)h * F + f) * P + k];
        if (p >= 0 && p < P) {
          ku = *reinterpret_cast<const uint2*>(k_p + ((size_t)h * P + p) * kD + lane * 4);
          vu = *reinterpret_cast<const uint2*>(v_p + ((size_t)h * P + p) * kD + lane * 4);
        } else {
          bad = true;
        }
      }
      *reinterpret_cast<uint2*>(kc + dst) = ku;
      *reinterpret_cast<uint2*>(vc + dst) = vu;
    }
    if (bad && lane == 0) status_set(st, FASTAR_ERR_DEVICE_ARG);
  }
  pdl_trigger();
}

// AnnCA: grid (query tiles, frames, heads); AnnSA: grid (query tiles,
// tables, heads).
// kRuns (AnnSA over a description of at most two buckets in one table, i.e.
// dense attention, dense denoising steps and the quantised matcher): tiles of
// consecutive slots are loaded as 64-row boxes (mapK64 / mapV64).  The
// bucketed form is compiled without that path, which would cost its gathers
// about 4 % even where it is never taken.
template <bool kSA, bool kRuns>
__global__ void __launch_bounds__(kThreads, 2) attn_tc_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                             const __grid_constant__ CUtensorMap mapK,
                                                             const __grid_constant__ CUtensorMap mapV,
                                                             const __grid_constant__ CUtensorMap mapK64,
                                                             const __grid_constant__ CUtensorMap mapV64, int H,
                                                             int Nq, float scale, CaArgs ca, SaArgs sa,
                                                             int32_t* st) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  if (block_status_bad(st)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.x * kM;
  const int h = blockIdx.z;
  const int g = blockIdx.y;  // AnnCA: frame
  const int kT = kSA ? (int)blockIdx.y : 0;  // AnnSA: table (the earlier tables' collisions are excluded)
  const float scale2 = scale * kLog2e;

  if (tid == 0) {
    tc::mbar_init(&sm.bar_q, kSA ? 128 : 1);  // AnnSA: every softmax thread gathers its query row
    for (int s = 0; s < kStages; ++s) {
      // one arrival with the TMA bytes (AnnSA: after the tile's metadata)
      tc::mbar_init(&sm.kfull[s], 1);
      tc::mbar_init(&sm.vfull[s], 1);
      tc::mbar_init(&sm.kempty[s], 1);     // QK commit
      tc::mbar_init(&sm.vempty[s], 1);     // PV commit (also: O holds this tile's product)
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&sm.sfull[b], 1);      // QK commit
      tc::mbar_init(&sm.pready[b], 4);     // softmax warps (P written to TMEM)
    }
    tc::mbar_init(&sm.odone, 1);           // commit after the last PV
    tc::mbar_init(&sm.fin, 1);             // last commit of the MMA issuer
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem, 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;  // S / P buffers at columns 0 and 64, O at 128
  bool ok = true;
  bool bad_index = false;

  // ---- AnnSA: the softmax threads gather their query rows right away
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;  // softmax warps: query row of the tile = TMEM lane
  int my_row = -1;
  if constexpr (kSA) {
    if (warp >= 2) {
      if (m0 + r < Nq) {
        const int x = sa.q_perm[((size_t)h * sa.T + kT) * Nq + m0 + r];
        if (x >= 0 && x < Nq) my_row = x; else bad_index = true;
      }
      const uint32_t q0 = tc::smem_u32(sm.Q);
      const char* src = my_row >= 0 ? (const char*)(sa.q + ((size_t)h * Nq + my_row) * kD) : (const char*)sa.q;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch)
        tc::cp_async16(q0 + tc::sw128_offset(r, ch, kM), src + (my_row >= 0 ? ch * 16 : 0), my_row >= 0 ? 16u : 0u);
      tc::cp_async_arrive_noinc(&sm.bar_q);
    }
  } else {
    if (warp >= 2 && m0 + r < ca.n_f) my_row = g * ca.n_f + m0 + r;
  }

  // ---- the key list of this CTA (every thread computes it)
  int nkeys = 0, kbeg = 0, n_live = 0;
  const int32_t* toff = nullptr;  // AnnSA: cache CSR offsets of table kT
  if constexpr (!kSA) {
    nkeys = min(max(ca.kept_cnt[(size_t)h * ca.F + g], 0), ca.P);
  } else {
    const int32_t* qp = sa.q_perm + ((size_t)h * sa.T + kT) * Nq;
    const int nrow = min(kM, Nq - m0);
    const int first = qp[m0], last = qp[m0 + nrow - 1];
    const uint32_t c_lo = (first >= 0 && first < Nq) ? sa.q_codes[((size_t)h * sa.T + kT) * Nq + first] : 0u;
    const uint32_t c_hi = (last >= 0 && last < Nq) ? sa.q_codes[((size_t)h * sa.T + kT) * Nq + last] : 0u;
    n_live = min(max(sa.size[h], 0), sa.C);
    toff = sa.offsets + ((size_t)h * sa.T + kT) * (sa.nb + 1);
    if (c_lo < (uint32_t)sa.nb && c_hi < (uint32_t)sa.nb && c_lo <= c_hi) {
      kbeg = min(max(toff[c_lo], 0), n_live);
      nkeys = min(max(toff[c_hi + 1], kbeg), n_live) - kbeg;
    } else {
      bad_index = true;
    }
  }
  const int ntiles = (nkeys + kN - 1) / kN;
  int issued_k = 0, issued_v = 0;  // producer: key / value tiles whose loads were issued

  if (warp == 0) {
    // ================================================= producer
    if constexpr (!kSA) {
      if (ntiles > 0 && lane == 0) {
        tc::prefetch_tensormap(&mapQ);
        tc::mbar_arrive_expect_tx(&sm.bar_q, kM * kD * 2);
        const int row0 = h * Nq + g * ca.n_f + m0;
        tc::tma_load_2d(sm.Q, &mapQ, &sm.bar_q, 0, row0);
        tc::tma_load_2d(sm.Q + kM * 128, &mapQ, &sm.bar_q, 64, row0);
      }
    }
    // row sources of tile j, rows lane and lane + 32 (AnnCA: prompt ids;
    // AnnSA: slots).  The loads are only issued here; the values are checked
    // when the next tile becomes current, so the warp does not wait for them.
    constexpr int kNoRow = INT_MIN;
    const int lim = kSA ? sa.C : ca.P;
    auto fetch_src = [&](int j, int* out) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int k = j * kN + lane + 32 * u;
        out[u] = kNoRow;
        if (k < nkeys) {
          if constexpr (!kSA) out[u] = ca.kept_idx[((size_t)h * ca.F + g) * ca.P + k];
          else out[u] = sa.perm[((size_t)h * sa.T + kT) * sa.C + kbeg + k];
        }
      }
    };
    auto check_src = [&](int* v) {
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (v[u] != kNoRow && (v[u] < 0 || v[u] >= lim)) {
          bad_index = true;
          v[u] = kNoRow;
        }
    };
    // AnnSA metadata of those rows: codes of the earlier tables and the
    // group counts m (log2 m is taken when the metadata is stored)
    uint32_t kc[kMaxT - 1][2];
    int mraw[2];
    auto fetch_meta = [&](const int* src) {
      if constexpr (kSA) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
#pragma unroll
          for (int w = 0; w < kMaxT - 1; ++w)
            kc[w][u] = (w < kT && src[u] >= 0) ? sa.codes[((size_t)h * sa.T + w) * sa.C + src[u]] : 0xfffffffeu;
          mraw[u] = src[u] >= 0 ? sa.m[(size_t)h * sa.C + src[u]] : 0;
        }
      }
    };
    const size_t rows_per_head = kSA ? (size_t)sa.C : (size_t)ca.P;
    // Key and value gathers advance independently: the key rows of tile j go
    // into key stage j % kStages once QK_{j-2} has freed it, the value rows
    // and metadata into value stage j % kStages once PV_{j-2} has.  Each side
    // keeps its own row sources, fetched one tile ahead.
    // AnnSA: the 64 rows of a key or value tile gathered by TMA, four rows
    // per tile::gather4 (one-row-high boxes of 64 columns): lane l fetches
    // rows 4 (l % 16) .. + 3 of column half l / 16.  Rows past the key list
    // read slot 0 (always a row of the tensor; those columns are masked).
    // A tile whose 64 slots are one run of consecutive rows of the head (a
    // one-bucket description of the cache) comes as two 64-row boxes
    // instead of 32 four-row gathers.  The test is taken for every tile only
    // in CTAs whose first tile is such a run (elsewhere runs are rare and the
    // test costs more than it saves), when the tile's slots are checked,
    // ahead of its gather.
    bool runs = false;
    auto is_run = [&](const int* src) -> bool {
      if (!kRuns || !runs) return false;
      const int base = __shfl_sync(0xffffffffu, src[0], 0);
      return __all_sync(0xffffffffu, base >= 0 && base + kN <= (int)rows_per_head && src[0] == base + lane &&
                                         src[1] == base + 32 + lane);
    };
    auto gather = [&](uint8_t* tile, const CUtensorMap* map, const CUtensorMap* map64, uint64_t* bar,
                      const int* src, bool run) {
      if constexpr (kRuns) {
        if (run) {
          const int y = (int)((size_t)h * rows_per_head) + __shfl_sync(0xffffffffu, src[0], 0);
          __syncwarp();  // the metadata stores, before lane 0's arrival
          if (lane == 0) {
            tc::mbar_arrive_expect_tx(bar, kN * kD * 2);
            tc::tma_load_2d(tile, map64, bar, 0, y);
            tc::tma_load_2d(tile + kN * 128, map64, bar, 64, y);
          }
          return;
        }
      }
      const int r0 = 4 * (lane & 15), hf = lane >> 4;
      int ys[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = r0 + e;
        const int a = __shfl_sync(0xffffffffu, src[0], r & 31);
        const int b = __shfl_sync(0xffffffffu, src[1], r & 31);
        const int sr = (r >> 5) ? b : a;
        ys[e] = (int)((size_t)h * rows_per_head) + (sr >= 0 ? sr : 0);
      }
      // every lane's metadata stores are ordered before lane 0's arrival
      // (a complete_tx that lands before the expect_tx is allowed)
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_expect_tx(bar, kN * kD * 2);
      tc::tma_gather4_2d(tile + hf * (kN * 128) + r0 * 128, map, bar, hf * 64, ys[0], ys[1], ys[2], ys[3]);
    };
    int ksrc[2] = {kNoRow, kNoRow}, knext[2] = {kNoRow, kNoRow}, vsrc[2] = {kNoRow, kNoRow},
        vnext[2] = {kNoRow, kNoRow};
    bool krun = false, vrun = false;
    if (lane == 0) {
      tc::prefetch_tensormap(&mapK);
      tc::prefetch_tensormap(&mapV);
      if constexpr (!kSA) {  // AnnCA: the prompt's own rows
        tc::prefetch_tensormap(&mapK64);
        tc::prefetch_tensormap(&mapV64);
      }
    }
    if constexpr (kSA) {
      fetch_src(0, ksrc);
      check_src(ksrc);
      runs = kRuns;
      krun = is_run(ksrc);
      runs = krun;
      vrun = krun;
      if (runs && lane == 0) {
        tc::prefetch_tensormap(&mapK64);
        tc::prefetch_tensormap(&mapV64);
      }
      vsrc[0] = ksrc[0];
      vsrc[1] = ksrc[1];
      fetch_meta(vsrc);
      if (ntiles > 1) {
        fetch_src(1, knext);
        fetch_src(1, vnext);
      }
    }
    int jk = 0, jv = 0;
    uint32_t idle = 0;
    while (ok && jv < ntiles) {
      bool did = false;
      if (jk < ntiles) {
        const int s = jk % kStages;
        int ready = 1;
        if (jk >= kStages)
          ready = lane == 0 ? (int)tc::mbar_test_wait(&sm.kempty[s], (uint32_t)((jk / kStages) - 1) & 1u) : 0;
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          if constexpr (!kSA) {
            if (lane == 0) {
              // every prompt token kept (the kept list is the prompt in
              // order): the prompt's own rows (mapK64); else the compacted ones
              const bool all = nkeys == ca.P;
              const int row = all ? h * ca.P + jk * kN : (h * ca.F + g) * ca.P64 + jk * kN;
              const CUtensorMap* map = all ? &mapK64 : &mapK;
              tc::mbar_arrive_expect_tx(&sm.kfull[s], kN * kD * 2);
              tc::tma_load_2d(sm.K[s], map, &sm.kfull[s], 0, row);
              tc::tma_load_2d(sm.K[s] + kN * 128, map, &sm.kfull[s], 64, row);
            }
          } else {
            gather(sm.K[s], &mapK, &mapK64, &sm.kfull[s], ksrc, krun);
          }
          ++jk;
          if constexpr (kSA) {
            ksrc[0] = knext[0];
            ksrc[1] = knext[1];
            check_src(ksrc);
            krun = is_run(ksrc);
            knext[0] = knext[1] = kNoRow;
            if (jk + 1 < ntiles) fetch_src(jk + 1, knext);
          }
          did = true;
        }
      }
      if (jv < jk) {
        const int s = jv % kStages;
        int ready = 1;
        if (jv >= kStages)
          ready = lane == 0 ? (int)tc::mbar_test_wait(&sm.vempty[s], (uint32_t)((jv / kStages) - 1) & 1u) : 0;
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          if constexpr (kSA) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
#pragma unroll
              for (int w = 0; w < kMaxT - 1; ++w)
                if (w < kT) sm.kcodes[s][w][lane + 32 * u] = kc[w][u];
              sm.bias[s][lane + 32 * u] = vsrc[u] >= 0 ? log2f((float)max(mraw[u], 1)) : 0.f;
            }
          }
          if constexpr (!kSA) {
            if (lane == 0) {
              const bool all = nkeys == ca.P;
              const int row = all ? h * ca.P + jv * kN : (h * ca.F + g) * ca.P64 + jv * kN;
              const CUtensorMap* map = all ? &mapV64 : &mapV;
              tc::mbar_arrive_expect_tx(&sm.vfull[s], kN * kD * 2);
              tc::tma_load_2d(sm.V[s], map, &sm.vfull[s], 0, row);
              tc::tma_load_2d(sm.V[s] + kN * 128, map, &sm.vfull[s], 64, row);
            }
          } else {
            // the metadata written above are published by the arrival that
            // carries the gather's bytes (after the warp barrier in gather)
            gather(sm.V[s], &mapV, &mapV64, &sm.vfull[s], vsrc, vrun);
          }
          ++jv;
          if constexpr (kSA) {
            vsrc[0] = vnext[0];
            vsrc[1] = vnext[1];
            check_src(vsrc);
            vrun = is_run(vsrc);
            if (jv < ntiles) fetch_meta(vsrc);  // lands while tile jv - 1 is consumed
            vnext[0] = vnext[1] = kNoRow;
            if (jv + 1 < ntiles) fetch_src(jv + 1, vnext);
          }
          did = true;
        }
      }
      if (did) {
        idle = 0;
      } else if (++idle > kIdlePolls) {
        ok = false;
      } else {
        __nanosleep(32);
      }
    }
    issued_k = jk;
    issued_v = jv;
  } else if (warp == 1) {
    // ================================================= MMA issuer
    // Issues QK_j (S_j = Q K_j^T into TMEM buffer j & 1) and PV_j (O += P_j
    // V_j, P_j read from the same TMEM buffer, where the softmax wrote it
    // over S_j) in whichever order their inputs become ready, with QK at
    // most one tile ahead of PV: QK_{j+2} is issued after PV_j, and the MMAs
    // of one thread run in issue order, so it cannot overwrite P_j early.
    constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kM, kN, 0, 0);
    constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kM, kD, 0, 1);
    if (ntiles > 0) ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.bar_q, 0));
    int jq = 0, jp = 0;
    uint32_t idle = 0;
    while (ok && jp < ntiles) {
      bool did = false;
      if (jp < jq) {
        const int s = jp % kStages, b = jp & 1;
        int ready = 0;
        if (lane == 0)
          ready = tc::mbar_test_wait(&sm.pready[b], (uint32_t)(jp >> 1) & 1u) &&
                  tc::mbar_test_wait(&sm.vfull[s], (uint32_t)(jp / kStages) & 1u);
        ready = __shfl_sync(0xffffffffu, ready, 0);
        if (ready) {
          tc::fence_proxy_async_smem();
          tc::tc_fence_after();
          if (lane == 0) {
            const uint32_t v0 = tc::smem_u32(sm.V[s]);
#pragma unroll
            for (int kk = 0; kk < kN / 16; ++kk)
              tc::mma_bf16_tmem_a(tmem + 128, tmem + b * kN + kk * 8,
                                  tc::sdesc_mnmajor_sw128(v0 + kk * 16 * 128, kN * 128), idesc_pv,
                                  (jp > 0 || kk > 0) ? 1u : 0u);
            tc::mma_commit(&sm.vempty[s]);
            if (jp == ntiles - 1) tc::mma_commit(&sm.odone);
          }
          __syncwarp();
          ++jp;
          did = true;
        }
      }
      if (!did && jq < ntiles && jq <= jp + 1) {
        const int s = jq % kStages, b = jq & 1;
        int ready = lane == 0 ? (int)tc::mbar_test_wait(&sm.kfull[s], (uint32_t)(jq / kStages) & 1u) : 0;
        ready = __shfl_sync(0xffffffffu, ready, 0);
        if (ready) {
          tc::fence_proxy_async_smem();
          tc::tc_fence_after();
          if (lane == 0) {
            const uint32_t q0 = tc::smem_u32(sm.Q), k0 = tc::smem_u32(sm.K[s]);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t oq = (kk >> 2) * kM * 128 + (kk & 3) * 32;
              const uint32_t okk = (kk >> 2) * kN * 128 + (kk & 3) * 32;
              tc::mma_bf16(tmem + b * kN, tc::sdesc_kmajor_sw128(q0 + oq), tc::sdesc_kmajor_sw128(k0 + okk),
                           idesc_qk, kk > 0 ? 1u : 0u);
            }
            tc::mma_commit(&sm.sfull[b]);
            tc::mma_commit(&sm.kempty[s]);
          }
          __syncwarp();
          ++jq;
          did = true;
        }
      }
      if (did) {
        idle = 0;
      } else if (++idle > kIdlePolls) {
        ok = false;
      } else {
        __nanosleep(32);
      }
    }
    // every MMA this warp issued has finished before TMEM is freed (also on
    // an expired wait, where nobody else may wait for them)
    if (jq > 0) {
      if (lane == 0) tc::mma_commit(&sm.fin);
      __syncwarp();
      if (!tc::mbar_wait(&sm.fin, 0)) ok = false;
    }
  } else {
    // ================================================= softmax (warps 2-5)
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    uint32_t qprev[kMaxT - 1] = {0xffffffffu, 0xffffffffu, 0xffffffffu};
    // keys of this row's bucket in table kT, in CTA key coordinates
    int run_a = 0, run_b = nkeys;
    if constexpr (kSA) {
      run_b = 0;
      if (my_row >= 0) {
#pragma unroll
        for (int w = 0; w < kMaxT - 1; ++w)
          if (w < kT) qprev[w] = sa.q_codes[((size_t)h * sa.T + w) * Nq + my_row];
        const uint32_t qk = sa.q_codes[((size_t)h * sa.T + kT) * Nq + my_row];
        if (qk < (uint32_t)sa.nb) {
          const int a = min(max(toff[qk], 0), n_live);
          const int b = min(max(toff[qk + 1], a), n_live);
          run_a = min(max(a - kbeg, 0), nkeys);
          run_b = min(max(b - kbeg, run_a), nkeys);
        } else {
          bad_index = true;
        }
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int s = j % kStages, b = j & 1;
      if constexpr (kSA) ok = tc::mbar_wait(&sm.vfull[s], (uint32_t)(j / kStages) & 1u);  // metadata
      ok = ok && tc::mbar_wait(&sm.sfull[b], (uint32_t)(j >> 1) & 1u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc::tc_fence_after();
      const uint64_t run = range_bits(run_a - j * kN, run_b - j * kN);
      uint32_t bits[2] = {(uint32_t)run, (uint32_t)(run >> 32)};
      if constexpr (kSA) {
        if (sa.row_mask && my_row >= 0) {
          const uint32_t* mw = sa.row_mask + ((size_t)h * Nq + my_row) * sa.mask_words;
          const int w0 = (kbeg + j * kN) >> 5;  // kbeg = 0 with the one-bucket description
#pragma unroll
          for (int q = 0; q < 2; ++q) bits[q] &= (w0 + q < sa.mask_words) ? mw[w0 + q] : 0u;
        }
      }
      bool live[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) live[q] = __any_sync(0xffffffffu, bits[q] != 0u);
      float v[2][32];
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (live[q]) tc::tmem_ld32(tmem + lane_base + b * kN + q * 32, v[q]);
      // scores in log2 units (masked: -inf) and their maximum; AnnCA keeps
      // the raw products and scales the maximum (scale > 0)
      float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (!live[q]) continue;
        if constexpr (kSA) {
          // drop slots an earlier table already admitted for this query
#pragma unroll
          for (int w = 0; w < kMaxT - 1; ++w) {
            if (w < kT && bits[q]) {
#pragma unroll
              for (int i4 = 0; i4 < 8; ++i4) {
                const uint4 c4 = *reinterpret_cast<const uint4*>(&sm.kcodes[s][w][q * 32 + i4 * 4]);
                const uint32_t eq = (c4.x == qprev[w] ? 1u : 0u) | (c4.y == qprev[w] ? 2u : 0u) |
                                    (c4.z == qprev[w] ? 4u : 0u) | (c4.w == qprev[w] ? 8u : 0u);
                bits[q] &= ~(eq << (i4 * 4));
              }
            }
          }
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 b4 = *reinterpret_cast<const float4*>(&sm.bias[s][q * 32 + i4 * 4]);
            const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = i4 * 4 + e;
              const float sc = ((bits[q] >> i) & 1u) ? fmaf(v[q][i], scale2, bb[e]) : -INFINITY;
              v[q][i] = sc;
              tm[e] = fmaxf(tm[e], sc);
            }
          }
        } else {
          if (!__all_sync(0xffffffffu, bits[q] == 0xffffffffu)) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[q][i] = ((bits[q] >> i) & 1u) ? v[q][i] : -INFINITY;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) tm[i & 3] = fmaxf(tm[i & 3], v[q][i]);
        }
      }
      float tmax = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3]));
      if constexpr (!kSA) tmax *= scale2;
      // raise the running max (and rescale O) only for a large increase
      const bool raise = tmax > m_run + kRescale;
      const float m_new = raise ? tmax : m_run;
      const float alpha = (raise && m_run != -INFINITY) ? exp2f(m_run - m_new) : 1.f;
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // wait until O holds P_0 V_0 .. P_{j-1} V_{j-1}
        ok = __all_sync(0xffffffffu, wait_pv(sm, j - 1));
        if (!ok) break;
        tc::tc_fence_after();
#pragma unroll
        for (int q = 0; q < kD / 32; ++q) {
          float o[32];
          tc::tmem_ld32(tmem + lane_base + 128 + q * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tc::tmem_st32(tmem + lane_base + 128 + q * 32, o);
        }
      }
      l_run *= alpha;
      m_run = m_new;
      // P_j (bf16 pairs, 32 columns) over S_j in TMEM; masked scores are
      // -inf and give 0 (scale > 0)
      const float m_sub = m_run == -INFINITY ? 0.f : m_run;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t packed_all[32];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t* packed = packed_all + 16 * q;
        if (live[q]) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float p0, p1;
            if constexpr (kSA) {
              p0 = ex2(v[q][i] - m_sub);
              p1 = ex2(v[q][i + 1] - m_sub);
            } else {
              p0 = ex2(fmaf(v[q][i], scale2, -m_sub));
              p1 = ex2(fmaf(v[q][i + 1], scale2, -m_sub));
            }
            ps[i & 3] += p0;
            ps[(i & 3) + 1] += p1;
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            packed[i >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) packed[i] = 0u;
        }
      }
      tc::tmem_st32u(tmem + lane_base + b * kN, packed_all);
      const float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
      l_run += psum;
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.pready[b]);
    }
    // ---- output: O (TMEM) staged per warp through shared memory (Q and K
    // are free once the last PV product has landed), then written one row
    // per warp instruction
    if (ok && ntiles > 0) {
      ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.odone, 0));  // the last PV product
      tc::tc_fence_after();
    }
    if constexpr (kSA) tc::cp_async_wait_all();  // the query rows (no key tile may have waited for them)
    if (ok) {
      uint8_t* wbase = sm.Q + quarter * (32 * kD * 4);
      if constexpr (kSA) {
        // fp32 rows of 512 bytes; chunk i of row `lane` at position (i + lane) % 32
#pragma unroll
        for (int q = 0; q < kD / 32; ++q) {
          float o[32];
          if (ntiles > 0) {
            tc::tmem_ld32(tmem + lane_base + 128 + q * 32, o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.f;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(wbase + lane * 512 + (((q * 8 + k) + lane) & 31) * 16) =
                make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
        __syncwarp();
        const size_t ri = (size_t)h * Nq + my_row;
        if (sa.T == 1 && !sa.parts_only) {
          // a single table: the partial is the result
          const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
          if (my_row >= 0 && sa.lse) sa.lse[ri] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
          for (int rr = 0; rr < 32; ++rr) {
            const int row = __shfl_sync(0xffffffffu, my_row, rr);
            const float iv = __shfl_sync(0xffffffffu, inv, rr);
            if (row < 0) continue;
            const float4 x = *reinterpret_cast<const float4*>(wbase + rr * 512 + ((lane + rr) & 31) * 16);
            const __nv_bfloat162 b0 = __floats2bfloat162_rn(x.x * iv, x.y * iv);
            const __nv_bfloat162 b1 = __floats2bfloat162_rn(x.z * iv, x.w * iv);
            uint2 u;
            u.x = *reinterpret_cast<const uint32_t*>(&b0);
            u.y = *reinterpret_cast<const uint32_t*>(&b1);
            *reinterpret_cast<uint2*>(sa.out + ((size_t)h * Nq + row) * kD + lane * 4) = u;
          }
        } else {
          // this table's partial, normalised by its own sum and stored in
          // fp16 (a convex combination of value rows, so well inside fp16's
          // range); the combine kernel weighs the tables by their sums
          const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
          for (int rr = 0; rr < 32; ++rr) {
            const int row = __shfl_sync(0xffffffffu, my_row, rr);
            const float iv = __shfl_sync(0xffffffffu, inv, rr);
            if (row < 0) continue;
            const float4 x = *reinterpret_cast<const float4*>(wbase + rr * 512 + ((lane + rr) & 31) * 16);
            const __half2 h0 = __floats2half2_rn(x.x * iv, x.y * iv);
            const __half2 h1 = __floats2half2_rn(x.z * iv, x.w * iv);
            uint2 u;
            u.x = *reinterpret_cast<const uint32_t*>(&h0);
            u.y = *reinterpret_cast<const uint32_t*>(&h1);
            *reinterpret_cast<uint2*>(sa.ws_o + (((size_t)(sa.slot0 + kT) * H + h) * Nq + row) * kD + lane * 4) = u;
          }
          if (my_row >= 0)
            sa.ws_ml[((size_t)(sa.slot0 + kT) * H + h) * Nq + my_row] = make_float2(l_run > 0.f ? m_run : -INFINITY, l_run);
        }
      } else {
        // normalised bf16 rows of 256 bytes; chunk i of row `lane` at position (i + lane) % 16
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int q = 0; q < kD / 32; ++q) {
          float o[32];
          if (ntiles > 0) {
            tc::tmem_ld32(tmem + lane_base + 128 + q * 32, o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.f;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 pb = __floats2bfloat162_rn(o[8 * k + 2 * e] * inv, o[8 * k + 2 * e + 1] * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&pb);
            }
            *reinterpret_cast<uint4*>(wbase + lane * 256 + (((q * 4 + k) + lane) & 15) * 16) = u;
          }
        }
        __syncwarp();
        for (int rr = 0; rr < 32; rr += 2) {
          const int rw = rr + (lane >> 4), c = lane & 15;
          const int row = __shfl_sync(0xffffffffu, my_row, rw);
          if (row < 0) continue;
          const uint4 x = *reinterpret_cast<const uint4*>(wbase + rw * 256 + ((c + rw) & 15) * 16);
          *reinterpret_cast<uint4*>(ca.out + ((size_t)h * Nq + row) * kD + c * 8) = x;
        }
      }
    }
  }
  if (bad_index) status_set(st, FASTAR_ERR_DEVICE_ARG);
  if (!ok) status_set(st, FASTAR_ERR_TIMEOUT);
  if (warp == 0) {
    // the producer's copies have landed before the CTA exits (also when a
    // wait elsewhere ran out and nobody consumed the last tiles): the last
    // kStages key and value loads are waited for, with the bounded wait
    tc::cp_async_wait_all();
    if (!kSA && ntiles > 0 && lane == 0 && !tc::mbar_wait(&sm.bar_q, 0)) status_set(st, FASTAR_ERR_TIMEOUT);
    if (lane == 0) {
      for (int t = max(0, issued_k - kStages); t < issued_k; ++t)
        if (!tc::mbar_wait(&sm.kfull[t % kStages], (uint32_t)(t / kStages) & 1u)) status_set(st, FASTAR_ERR_TIMEOUT);
      for (int t = max(0, issued_v - kStages); t < issued_v; ++t)
        if (!tc::mbar_wait(&sm.vfull[t % kStages], (uint32_t)(t / kStages) & 1u)) status_set(st, FASTAR_ERR_TIMEOUT);
    }
    __syncwarp();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 256);
  pdl_trigger();
}

// Merge the T per-table partials of each query: a warp handles kCombineQ
// queries, four dimensions per lane; every (max, sum) and partial row of its
// queries is loaded before any is used.  Compiled for the number of partials
// (kT = 2, the workloads' two tables, or up to four), so that a warp holds
// only the partials there are: four queries per warp (two with up to four
// partials, within the register budget) at four CTAs per SM.
template <int kT, int kCombineQ>
__global__ void __launch_bounds__(256, 4) annsa_combine_kernel(const __half* __restrict__ ws_o,
                                                            const float2* __restrict__ ws_ml, int T, int H,
                                                            int Nq, __nv_bfloat16* __restrict__ out,
                                                            float* __restrict__ lse, int32_t* st) {
  constexpr int kMaxT = kT;  // partials held per query
  pdl_wait();
  if (status_bad(st)) return;
  const int h = blockIdx.y;
  const int i0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * kCombineQ;
  const int lane = threadIdx.x & 31;
  float2 ml[kCombineQ][kMaxT];
  uint2 o[kCombineQ][kMaxT];
#pragma unroll
  for (int k = 0; k < kCombineQ; ++k) {
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      ml[k][t] = make_float2(-INFINITY, 0.f);
      o[k][t] = make_uint2(0u, 0u);
      if (t < T && i0 + k < Nq) {
        const size_t r = ((size_t)t * H + h) * Nq + i0 + k;
        ml[k][t] = __ldcs(ws_ml + r);
        o[k][t] = __ldcs(reinterpret_cast<const uint2*>(ws_o + r * kD) + lane);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kCombineQ; ++k) {
    const int i = i0 + k;
    if (i >= Nq) break;
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) M = fmaxf(M, ml[k][t].x);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      // weight of table t's normalised partial: its sum on the common scale
      const float w = ml[k][t].x == -INFINITY ? 0.f : exp2f(ml[k][t].x - M) * ml[k][t].y;
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&o[k][t].x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&o[k][t].y));
      L += w;
      acc.x = fmaf(a.x, w, acc.x);
      acc.y = fmaf(a.y, w, acc.y);
      acc.z = fmaf(b.x, w, acc.z);
      acc.w = fmaf(b.y, w, acc.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 b1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&b0);
    u.y = *reinterpret_cast<const uint32_t*>(&b1);
    *reinterpret_cast<uint2*>(out + ((size_t)h * Nq + i) * kD + lane * 4) = u;
    if (lse && lane == 0) lse[(size_t)h * Nq + i] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  pdl_trigger();
}

// mk64 / mv64: AnnSA's 64-row-box maps of the cache keys and values (for
// tiles of consecutive slots); AnnCA's maps of the prompt's keys and values
// (for the (head, frame)s that keep every prompt token).
template <bool kSA, bool kRuns = false>
int launch_attn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mk64,
                const CUtensorMap& mv64, dim3 grid, int H, int Nq, float scale, const CaArgs& ca, const SaArgs& sa,
                int32_t* st, cudaStream_t s) {
  const size_t smem = sizeof(AttnSmem) + 1024;
  if (cudaFuncSetAttribute(attn_tc_kernel<kSA, kRuns>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_CUDA;
  }
  fastar::launch_pdl((attn_tc_kernel<kSA, kRuns>), grid, kThreads, smem, s, mq, mk, mv, mk64, mv64, H, Nq, scale, ca, sa,
                     st);
  FASTAR_LAUNCHED(s, kSA ? "annsa_tc" : "annca_tc");
  return FASTAR_OK;
}

int p64_of(int P) { return (P + kN - 1) / kN * kN; }

// AnnSA: the run-capable kernel for a description of at most two buckets in
// one table (dense attention, dense denoising steps), the bucketed one
// otherwise.
int sa_launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mk64,
              const CUtensorMap& mv64, dim3 grid, int H, int Nq, float scale, const CaArgs& ca, const SaArgs& sa,
              int32_t* st, cudaStream_t s) {
  if (sa.T == 1 && sa.nb <= 2) return launch_attn<true, true>(mq, mk, mv, mk64, mv64, grid, H, Nq, scale, ca, sa, st, s);
  return launch_attn<true, false>(mq, mk, mv, mk64, mv64, grid, H, Nq, scale, ca, sa, st, s);
}

// AnnSA: tensor maps of the cache's K and V ([H * C][D] bf16) with
// one-row-high boxes of 64 columns, for the producer's tile::gather4 loads,
// and with 64-row boxes, for tiles of consecutive slots.
int make_sa_maps(const fastar_cache* c, CUtensorMap* mk, CUtensorMap* mv, CUtensorMap* mk64, CUtensorMap* mv64) {
  const uint64_t rows = (uint64_t)c->H * (uint64_t)c->C;
  if (make_tmap_bf16_2d(mk, c->K, rows, kD, 1, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  if (make_tmap_bf16_2d(mv, c->V, rows, kD, 1, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  if (make_tmap_bf16_2d(mk64, c->K, rows, kD, kN, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  if (make_tmap_bf16_2d(mv64, c->V, rows, kD, kN, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  return FASTAR_OK;
}

}  // namespace

size_t annsa_tc_ws_bytes(int H, int Nq, int D, int T) {
  if (D != kD || T > kMaxT) return 0;
  if (T == 1) return 0;  // a single table writes the output directly
  const size_t o = (size_t)T * H * Nq * kD * sizeof(__half);
  const size_t ml = (size_t)T * H * Nq * sizeof(float2);
  return ((o + 255) & ~(size_t)255) + ((ml + 255) & ~(size_t)255);
}

size_t annca_tc_ws_bytes(int H, int F, int P, int D) {
  if (D != kD) return 0;
  const size_t half = (size_t)H * F * p64_of(P) * kD * sizeof(__nv_bfloat16);
  return 2 * ((half + 255) & ~(size_t)255);
}

int launch_annca_tc(fastar_dtype dt, const void* q, const void* k_p, const void* v_p,
                    const int32_t* kept_idx, const int32_t* kept_cnt, int H, int F, int n_f, int P, int D,
                    float scale, void* out, void* ws, size_t ws_bytes, int32_t* st, cudaStream_t s) {
  if (dt != FASTAR_BF16 || D != kD) return FASTAR_ERR_UNSUPPORTED;
  const int Nq = F * n_f;
  if (Nq == 0 || H == 0) return FASTAR_OK;
  const int P64 = p64_of(P);
  if (P64 == 0) {
    // no prompt tokens: every kept set is empty
    CUtensorMap mq;
    if (make_tmap_bf16_2d(&mq, q, (uint64_t)H * Nq, kD, kM, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
    CaArgs ca{(const __nv_bfloat16*)k_p, (const __nv_bfloat16*)v_p, kept_idx, kept_cnt, F, n_f, P, 0,
              (__nv_bfloat16*)out};
    SaArgs sa{};
    return launch_attn<false>(mq, mq, mq, mq, mq, dim3((n_f + kM - 1) / kM, F, H), H, Nq, scale, ca, sa, st, s);
  }
  if (!ws || ws_bytes < annca_tc_ws_bytes(H, F, P, D)) return FASTAR_ERR_WORKSPACE;
  const size_t half = (((size_t)H * F * P64 * kD * sizeof(__nv_bfloat16)) + 255) & ~(size_t)255;
  __nv_bfloat16* kc = (__nv_bfloat16*)ws;
  __nv_bfloat16* vc = (__nv_bfloat16*)((char*)ws + half);
  fastar::launch_pdl((annca_compact_kernel), dim3(P64 / kN, F, H), 256, 0, s, (const __nv_bfloat16*)k_p,
                     (const __nv_bfloat16*)v_p, kept_idx, kept_cnt, F, P, P64, kc, vc, st);
  FASTAR_LAUNCHED(s, "annca_compact");
  CUtensorMap mq, mk, mv, mkp, mvp;
  if (make_tmap_bf16_2d(&mq, q, (uint64_t)H * Nq, kD, kM, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  if (make_tmap_bf16_2d(&mk, kc, (uint64_t)H * F * P64, kD, kN, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  if (make_tmap_bf16_2d(&mv, vc, (uint64_t)H * F * P64, kD, kN, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  // the prompt itself, for the (head, frame)s that keep all of it
  if (make_tmap_bf16_2d(&mkp, k_p, (uint64_t)H * P, kD, kN, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  if (make_tmap_bf16_2d(&mvp, v_p, (uint64_t)H * P, kD, kN, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  CaArgs ca{(const __nv_bfloat16*)k_p, (const __nv_bfloat16*)v_p, kept_idx, kept_cnt, F, n_f, P, P64,
            (__nv_bfloat16*)out};
  SaArgs sa{};
  return launch_attn<false>(mq, mk, mv, mkp, mvp, dim3((n_f + kM - 1) / kM, F, H), H, Nq, scale, ca, sa, st, s);
}

int launch_annsa_tc(fastar_dtype dt, const void* q, const uint32_t* q_codes, const int32_t* q_perm,
                    const int32_t* q_offsets, int Nq, const fastar_cache* c, float scale, void* out,
                    float* lse, void* ws, int32_t* st, cudaStream_t s) {
  (void)q_offsets;
  if (dt != FASTAR_BF16 || c->D != kD || c->T > kMaxT) return FASTAR_ERR_UNSUPPORTED;
  if (Nq == 0 || c->H == 0) return FASTAR_OK;
  if (c->T > 1 && !ws) return FASTAR_ERR_WORKSPACE;
  const size_t o_bytes = ((size_t)c->T * c->H * Nq * kD * sizeof(__half) + 255) & ~(size_t)255;
  SaArgs sa{(const __nv_bfloat16*)q, q_codes, q_perm, (const __nv_bfloat16*)c->K,
            (const __nv_bfloat16*)c->V, c->m, c->codes, c->size, c->perm, c->offsets, c->C, c->T,
            1 << c->B, (__half*)ws, (float2*)((char*)ws + o_bytes), (__nv_bfloat16*)out, lse, 0, 0, nullptr, 0};
  CaArgs ca{};
  CUtensorMap dummy, mk, mv, mk64, mv64;
  memset(&dummy, 0, sizeof(dummy));
  if (make_sa_maps(c, &mk, &mv, &mk64, &mv64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  // every table in one launch: the tables' CTAs fill each other's waves
  const int rc = sa_launch(dummy, mk, mv, mk64, mv64, dim3((Nq + kM - 1) / kM, c->T, c->H), c->H, Nq, scale, ca,
                                   sa, st, s);
  if (rc != FASTAR_OK || c->T == 1) return rc;
  const int cq = c->T <= 2 ? 4 : 2;  // queries per warp of the combine kernel
  fastar::launch_pdl(c->T <= 2 ? annsa_combine_kernel<2, 4> : annsa_combine_kernel<4, 2>,
                     dim3((Nq + 8 * cq - 1) / (8 * cq), c->H), 256, 0, s, sa.ws_o, sa.ws_ml, c->T, c->H, Nq,
                                                                 (__nv_bfloat16*)out, lse, st);
  FASTAR_LAUNCHED(s, "annsa_combine");
  return FASTAR_OK;
}


// AnnSA over a one-table description of the keys with a per-query selection
// mask (the quantised matcher): the CTA writes the normalised output.
int launch_annsa_masked(fastar_dtype dt, const void* q, const uint32_t* q_codes, const int32_t* q_perm,
                        const int32_t* q_offsets, int Nq, const fastar_cache* c, float scale, void* out, float* lse,
                        const uint32_t* mask, int mask_words, int32_t* st, cudaStream_t s) {
  (void)q_offsets;
  if (dt != FASTAR_BF16 || c->D != kD || c->T != 1) return FASTAR_ERR_UNSUPPORTED;
  if (Nq == 0 || c->H == 0) return FASTAR_OK;
  SaArgs sa{(const __nv_bfloat16*)q, q_codes, q_perm, (const __nv_bfloat16*)c->K,
            (const __nv_bfloat16*)c->V, c->m, c->codes, c->size, c->perm, c->offsets, c->C, 1,
            1 << c->B, nullptr, nullptr, (__nv_bfloat16*)out, lse, 0, 0, mask, mask_words};
  CaArgs ca{};
  CUtensorMap dummy, mk, mv, mk64, mv64;
  memset(&dummy, 0, sizeof(dummy));
  if (make_sa_maps(c, &mk, &mv, &mk64, &mv64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  return launch_attn<true, true>(dummy, mk, mv, mk64, mv64, dim3((Nq + kM - 1) / kM, 1, c->H), c->H, Nq, scale, ca,
                                 sa, st, s);
}

size_t annsa_parts_ws_bytes(int H, int Nq, int D, int parts) {
  if (D != kD || parts < 1 || parts > kMaxT) return 0;
  const size_t o = (size_t)parts * H * Nq * kD * sizeof(__half);
  const size_t ml = (size_t)parts * H * Nq * sizeof(float2);
  return ((o + 255) & ~(size_t)255) + ((ml + 255) & ~(size_t)255);
}

// The partials of one AnnSA call for slots base .. base + T - 1 of a
// workspace of `parts` slots (no output), and the merge of all slots.
int launch_annsa_parts(const void* q, const uint32_t* q_codes, const int32_t* q_perm, int Nq,
                       const fastar_cache* c, float scale, int base, int parts, void* ws, int32_t* st,
                       cudaStream_t s) {
  if (c->dt != FASTAR_BF16 || c->D != kD) return FASTAR_ERR_UNSUPPORTED;
  if (Nq == 0 || c->H == 0) return FASTAR_OK;
  const size_t o_bytes = ((size_t)parts * c->H * Nq * kD * sizeof(__half) + 255) & ~(size_t)255;
  SaArgs sa{(const __nv_bfloat16*)q, q_codes, q_perm, (const __nv_bfloat16*)c->K,
            (const __nv_bfloat16*)c->V, c->m, c->codes, c->size, c->perm, c->offsets, c->C, c->T,
            1 << c->B, (__half*)ws, (float2*)((char*)ws + o_bytes), nullptr, nullptr, base, 1, nullptr, 0};
  CaArgs ca{};
  CUtensorMap dummy, mk, mv, mk64, mv64;
  memset(&dummy, 0, sizeof(dummy));
  if (make_sa_maps(c, &mk, &mv, &mk64, &mv64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  return sa_launch(dummy, mk, mv, mk64, mv64, dim3((Nq + kM - 1) / kM, c->T, c->H), c->H, Nq, scale, ca, sa,
                           st, s);
}

int launch_annsa_combine(int H, int Nq, int parts, const void* ws, void* out, float* lse, int32_t* st,
                         cudaStream_t s) {
  if (Nq == 0 || H == 0) return FASTAR_OK;
  const size_t o_bytes = ((size_t)parts * H * Nq * kD * sizeof(__half) + 255) & ~(size_t)255;
  const int cq = parts <= 2 ? 4 : 2;  // queries per warp of the combine kernel
  fastar::launch_pdl(parts <= 2 ? annsa_combine_kernel<2, 4> : annsa_combine_kernel<4, 2>,
                     dim3((Nq + 8 * cq - 1) / (8 * cq), H), 256, 0, s,
                     (const __half*)ws, (const float2*)((const char*)ws + o_bytes), parts, H, Nq,
                     (__nv_bfloat16*)out, lse, st);
  FASTAR_LAUNCHED(s, "annsa_combine");
  return FASTAR_OK;
}

}  // namespace fastar
