// AnnCA and AnnSA attention on the tensor cores (tcgen05 + TMEM, bf16).
//
// One CTA (4 warps, one thread per query row) owns 128 queries and walks
// their keys 128 at a time:
//   S = Q K^T            8 MMAs (M 128, N 128, K 16) into TMEM columns 0..127
//   softmax              each thread reads its row of S from TMEM, applies
//                        the scale, the + ln m bias and the mask, updates its
//                        running max / sum (base-2 online softmax) and writes
//                        P (bf16) into shared memory over the spent K tile
//   O_tile = P V         8 MMAs, V as an MN-major operand, TMEM columns
//                        128..255; the thread rescales its fp32 accumulator
//                        row in registers and adds O_tile.
// Keys and values are gathered row by row with cp.async into the 128-byte
// swizzled layout; the value tile uses the same physical layout, read by the
// MMA as an MN-major operand.
//
// AnnCA (gist.science technical summary 2.B): the CTA owns 128 queries of
// one frame (loaded by TMA, two 64-column boxes) and walks the frame's kept
// prompt tokens; it writes the normalised output.
// AnnSA (gist.science 2.C; paper.rainbus.top method steps; + ln m from
// paperlayer.ai appendix A, Lemma A.1): one launch per LSH table t.  The CTA
// owns 128 consecutive queries of the chunk in the bucket order of table t
// (the query CSR) and walks the cache slots of the buckets they span (the
// cache CSR, sorted by code too).  A slot is allowed for a query iff their
// table-t codes agree and no earlier table already allowed it, so every
// allowed pair is visited exactly once over the T tables.  Because both
// sides are bucket-sorted, a warp skips every 32-key chunk whose code range
// does not meet the code range of its 32 queries.  Each table writes an
// unnormalised partial (o, running max, sum); a combine kernel merges the T
// partials per query.
#include <math.h>

#include "common.cuh"
#include "tc.cuh"

namespace fastar {

namespace {

constexpr int kM = 128, kN = 128, kD = 128, kMaxT = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnSmem {
  uint8_t Q[kM * kD * 2];
  uint8_t K[kN * kD * 2];  // key tile, then P (bf16, K-major over keys)
  uint8_t V[kN * kD * 2];
  float bias[kN];
  uint32_t kcodes[kMaxT][kN];
  int rows[kM];
  uint64_t bar_q, bar_mma;
  uint32_t tmem;
};

struct CaArgs {
  const __nv_bfloat16* k_p;
  const __nv_bfloat16* v_p;
  const int32_t* kept_idx;
  const int32_t* kept_cnt;
  int F, n_f, P;
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
  float* ws_o;   // [T][H][Nq][D] unnormalised accumulators
  float2* ws_ml; // [T][H][Nq] (running max in log2 units, sum)
};

// One 128-key step of the online softmax for the calling thread's row.
// kT: AnnSA table (the mask compares kT + 1 codes); -1 for AnnCA.
// qlo/qhi: code range of the warp's queries in table kT (AnnSA).
// Returns false when a bounded wait expired.
template <int kT>
__device__ __forceinline__ bool attend_tile(AttnSmem& sm, uint32_t tmem, int nvalid, float scale2,
                                            const uint32_t* qcode, uint32_t qlo, uint32_t qhi, float& m_run,
                                            float& l_run, float* acc, uint32_t& phase, bool ok) {
  constexpr bool kSA = kT >= 0;
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kM, kN, 0, 0);
  constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kM, kD, 0, 1);
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (tid == 0 && ok) {
    const uint32_t q0 = tc::smem_u32(sm.Q), k0 = tc::smem_u32(sm.K);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t oq = (kk >> 2) * kM * 128 + (kk & 3) * 32;
      const uint32_t okk = (kk >> 2) * kN * 128 + (kk & 3) * 32;
      tc::mma_bf16(tmem, tc::sdesc_kmajor_sw128(q0 + oq), tc::sdesc_kmajor_sw128(k0 + okk), idesc_qk,
                   kk > 0 ? 1u : 0u);
    }
    tc::mma_commit(&sm.bar_mma);
  }
  if (ok) ok = tc::mbar_wait(&sm.bar_mma, phase);
  ok = __all_sync(0xffffffffu, ok);
  phase ^= 1;
  tc::tc_fence_after();

  // which 32-key chunks can hold an allowed key for some query of this warp
  bool live[kN / 32];
#pragma unroll
  for (int q = 0; q < kN / 32; ++q) {
    live[q] = q * 32 < nvalid;
    if constexpr (kSA) {
      if (live[q]) {
        const uint32_t klo = sm.kcodes[kT][q * 32];
        const uint32_t khi = sm.kcodes[kT][min(q * 32 + 31, nvalid - 1)];
        live[q] = !(khi < qlo || klo > qhi);
      }
    }
  }

  // pass 1: masked maximum of the row and the allowed bits
  uint32_t allow_bits[kN / 32];
  float tmax = -INFINITY;
#pragma unroll
  for (int q = 0; q < kN / 32; ++q) {
    allow_bits[q] = 0u;
    if (!ok || !live[q]) continue;
    float v[32];
    tc::tmem_ld32(tmem + lane_base + q * 32, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = q * 32 + i;
      bool allow = c < nvalid;
      float s = v[i] * scale2;
      if constexpr (kSA) {
        allow = allow && sm.kcodes[kT][c] == qcode[kT];
#pragma unroll
        for (int u = 0; u < kT; ++u) allow = allow && sm.kcodes[u][c] != qcode[u];
        s += sm.bias[c];
      }
      allow_bits[q] |= (allow ? 1u : 0u) << i;
      tmax = allow ? fmaxf(tmax, s) : tmax;
    }
  }
  const float m_new = fmaxf(m_run, tmax);
  const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
  // pass 2: P = 2^(s - m_new) written as bf16 over the spent key tile
  float psum = 0.f;
#pragma unroll
  for (int q = 0; q < kN / 32; ++q) {
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) packed[i] = 0u;
    if (ok && live[q]) {
      // the warp loads the chunk collectively, even for rows that allow nothing in it
      float v[32];
      tc::tmem_ld32(tmem + lane_base + q * 32, v);
      if (allow_bits[q]) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float p2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = q * 32 + i + e;
            float s = v[i + e] * scale2;
            if constexpr (kSA) s += sm.bias[c];
            p2[e] = ((allow_bits[q] >> (i + e)) & 1u) ? exp2f(s - m_new) : 0.f;
          }
          const __nv_bfloat162 b = __floats2bfloat162_rn(p2[0], p2[1]);
          psum += p2[0] + p2[1];
          packed[i >> 1] = *reinterpret_cast<const uint32_t*>(&b);
        }
      }
    }
    // 32 keys = 4 chunks of 8 keys; chunk index over 128 keys is q*4 + k
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 u = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
      *reinterpret_cast<uint4*>(sm.K + tc::sw128_offset(tid, q * 4 + k, kM)) = u;
    }
  }
  l_run = l_run * alpha + psum;
  m_run = m_new;
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (tid == 0 && ok) {
    const uint32_t p0 = tc::smem_u32(sm.K), v0 = tc::smem_u32(sm.V);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t op = (kk >> 2) * kM * 128 + (kk & 3) * 32;
      tc::mma_bf16(tmem + 128, tc::sdesc_kmajor_sw128(p0 + op),
                   tc::sdesc_mnmajor_sw128(v0 + kk * 16 * 128, kN * 128), idesc_pv, kk > 0 ? 1u : 0u);
    }
    tc::mma_commit(&sm.bar_mma);
  }
  if (ok) ok = tc::mbar_wait(&sm.bar_mma, phase);
  ok = __all_sync(0xffffffffu, ok);
  phase ^= 1;
  tc::tc_fence_after();
  if (ok) {
#pragma unroll
    for (int q = 0; q < kD / 32; ++q) {
      float v[32];
      tc::tmem_ld32(tmem + lane_base + 128 + q * 32, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[q * 32 + i] = fmaf(acc[q * 32 + i], alpha, v[i]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  return ok;
}

// kT = -1: AnnCA (grid: query tiles x frames x heads); kT >= 0: AnnSA table
// kT (grid: query tiles x 1 x heads).
template <int kT>
__global__ void __launch_bounds__(128) attn_tc_kernel(const __grid_constant__ CUtensorMap mapQ, int H,
                                                      int Nq, float scale, CaArgs ca, SaArgs sa,
                                                      int32_t* st) {
  constexpr bool kSA = kT >= 0;
  extern __shared__ uint8_t smem_raw[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  if (block_status_bad(st)) return;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int m0 = blockIdx.x * kM;
  const int h = blockIdx.z;
  const float scale2 = scale * kLog2e;

  if (tid == 0) {
    tc::mbar_init(&sm.bar_q, 1);
    tc::mbar_init(&sm.bar_mma, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem, 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;
  bool ok = true;
  bool bad_index = false;

  // ---- queries and the key list
  int nkeys = 0, kbeg = 0;
  uint32_t qcode[kMaxT] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
  uint32_t qlo = 0xffffffffu, qhi = 0u;
  int my_row = -1;  // query index of this thread's row (-1: padding)
  if constexpr (!kSA) {
    const int f = blockIdx.y;
    if (tid == 0) {
      tc::prefetch_tensormap(&mapQ);
      tc::mbar_arrive_expect_tx(&sm.bar_q, kM * kD * 2);
      const int row0 = h * Nq + f * ca.n_f + m0;
      tc::tma_load_2d(sm.Q, &mapQ, &sm.bar_q, 0, row0);
      tc::tma_load_2d(sm.Q + kM * 128, &mapQ, &sm.bar_q, 64, row0);
    }
    nkeys = min(max(ca.kept_cnt[(size_t)h * ca.F + f], 0), ca.P);
    if (m0 + tid < ca.n_f) my_row = f * ca.n_f + m0 + tid;
    ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.bar_q, 0));
  } else {
    const int32_t* qp = sa.q_perm + ((size_t)h * sa.T + kT) * Nq;
    const int nrow = min(kM, Nq - m0);
    if (tid < nrow) {
      const int qi = qp[m0 + tid];
      if (qi >= 0 && qi < Nq) my_row = qi; else bad_index = true;
    }
    sm.rows[tid] = my_row;
    __syncthreads();
    tc::gather_rows_sw128(tc::smem_u32(sm.Q), kM,
                          [&](int r) -> const void* {
                            const int qi = sm.rows[r];
                            return qi >= 0 ? (const void*)(sa.q + ((size_t)h * Nq + qi) * kD) : nullptr;
                          },
                          tid, 128, sa.q);
    tc::cp_async_commit();
#pragma unroll
    for (int u = 0; u <= kT; ++u)
      qcode[u] = my_row >= 0 ? sa.q_codes[((size_t)h * sa.T + u) * Nq + my_row] : 0xffffffffu;
    // code range of the warp's queries (padding rows excluded)
    uint32_t lo = my_row >= 0 ? qcode[kT] : 0xffffffffu, hi = my_row >= 0 ? qcode[kT] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    qlo = lo;
    qhi = hi;
    // key range: the cache buckets spanned by this tile's table-kT codes
    const int first = qp[m0], last = qp[m0 + nrow - 1];
    const uint32_t c_lo = (first >= 0 && first < Nq) ? sa.q_codes[((size_t)h * sa.T + kT) * Nq + first] : 0u;
    const uint32_t c_hi = (last >= 0 && last < Nq) ? sa.q_codes[((size_t)h * sa.T + kT) * Nq + last] : 0u;
    const int n_live = min(max(sa.size[h], 0), sa.C);
    if (c_lo < (uint32_t)sa.nb && c_hi < (uint32_t)sa.nb && c_lo <= c_hi) {
      const int32_t* off = sa.offsets + ((size_t)h * sa.T + kT) * (sa.nb + 1);
      kbeg = min(max(off[c_lo], 0), n_live);
      nkeys = min(max(off[c_hi + 1], kbeg), n_live) - kbeg;
    } else if (tid == 0) {
      bad_index = true;
    }
    tc::cp_async_wait_all();
  }

  float m_run = -INFINITY, l_run = 0.f;
  float acc[kD];
#pragma unroll
  for (int i = 0; i < kD; ++i) acc[i] = 0.f;
  uint32_t phase = 0;

  for (int k0 = 0; k0 < nkeys && ok; k0 += kN) {
    const int nvalid = min(kN, nkeys - k0);
    // row sources of this key tile (AnnCA: kept prompt ids; AnnSA: cache slots)
    int src = -1;
    if (tid < nvalid) {
      if constexpr (!kSA) {
        const int p = ca.kept_idx[((size_t)h * ca.F + blockIdx.y) * ca.P + k0 + tid];
        if (p >= 0 && p < ca.P) src = p; else bad_index = true;
      } else {
        const int s = sa.perm[((size_t)h * sa.T + kT) * sa.C + kbeg + k0 + tid];
        if (s >= 0 && s < sa.C) src = s; else bad_index = true;
      }
    }
    sm.rows[tid] = src;  // reuse: key source per row of this tile
    if constexpr (kSA) {
#pragma unroll
      for (int u = 0; u <= kT; ++u)
        sm.kcodes[u][tid] = src >= 0 ? sa.codes[((size_t)h * sa.T + u) * sa.C + src] : 0xfffffffeu;
      sm.bias[tid] = src >= 0 ? log2f((float)max(sa.m[(size_t)h * sa.C + src], 1)) : 0.f;
    }
    __syncthreads();
    const __nv_bfloat16* kbase = kSA ? sa.K : ca.k_p;
    const __nv_bfloat16* vbase = kSA ? sa.V : ca.v_p;
    const size_t rows_per_head = kSA ? (size_t)sa.C : (size_t)ca.P;
    auto krow = [&](int r) -> const void* {
      const int s = sm.rows[r];
      return s >= 0 ? (const void*)(kbase + ((size_t)h * rows_per_head + s) * kD) : nullptr;
    };
    auto vrow = [&](int r) -> const void* {
      const int s = sm.rows[r];
      return s >= 0 ? (const void*)(vbase + ((size_t)h * rows_per_head + s) * kD) : nullptr;
    };
    tc::gather_rows_sw128(tc::smem_u32(sm.K), kN, krow, tid, 128, kbase);
    tc::gather_rows_sw128(tc::smem_u32(sm.V), kN, vrow, tid, 128, vbase);
    tc::cp_async_commit();
    tc::cp_async_wait_all();
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    ok = attend_tile<kT>(sm, tmem, nvalid, scale2, qcode, qlo, qhi, m_run, l_run, acc, phase, ok);
  }

  if (bad_index) status_set(st, FASTAR_ERR_DEVICE_ARG);
  if (!ok) {
    if (tid == 0) status_set(st, FASTAR_ERR_TIMEOUT);
  } else if (my_row >= 0) {
    if constexpr (!kSA) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* o = ca.out + ((size_t)h * Nq + my_row) * kD;
#pragma unroll
      for (int i = 0; i < kD; i += 8) {
        uint4 u;
        uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(acc[i + 2 * e] * inv, acc[i + 2 * e + 1] * inv);
          w[e] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(o + i) = u;
      }
    } else {
      const size_t r = ((size_t)kT * H + h) * Nq + my_row;
      float* o = sa.ws_o + r * kD;
#pragma unroll
      for (int i = 0; i < kD; i += 4) *reinterpret_cast<float4*>(o + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
      sa.ws_ml[r] = make_float2(m_run, l_run);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// Merge the T per-table partials of each query (warp per query).
__global__ void __launch_bounds__(256) annsa_combine_kernel(const float* __restrict__ ws_o,
                                                            const float2* __restrict__ ws_ml, int T, int H,
                                                            int Nq, __nv_bfloat16* __restrict__ out,
                                                            float* __restrict__ lse, int32_t* st) {
  if (status_bad(st)) return;
  const int h = blockIdx.y;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= Nq) return;
  float M = -INFINITY;
  for (int t = 0; t < T; ++t) M = fmaxf(M, ws_ml[((size_t)t * H + h) * Nq + i].x);
  float L = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int t = 0; t < T; ++t) {
      const size_t r = ((size_t)t * H + h) * Nq + i;
      const float2 ml = ws_ml[r];
      if (ml.x == -INFINITY) continue;
      const float w = exp2f(ml.x - M);
      L = fmaf(ml.y, w, L);
      const float4 a = *reinterpret_cast<const float4*>(ws_o + r * kD + lane * 4);
      o.x = fmaf(a.x, w, o.x);
      o.y = fmaf(a.y, w, o.y);
      o.z = fmaf(a.z, w, o.z);
      o.w = fmaf(a.w, w, o.w);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* dst = out + ((size_t)h * Nq + i) * kD + lane * 4;
  const __nv_bfloat162 b0 = __floats2bfloat162_rn(o.x * inv, o.y * inv);
  const __nv_bfloat162 b1 = __floats2bfloat162_rn(o.z * inv, o.w * inv);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&b0);
  u.y = *reinterpret_cast<const uint32_t*>(&b1);
  *reinterpret_cast<uint2*>(dst) = u;
  if (lse && lane == 0) lse[(size_t)h * Nq + i] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

template <int kT>
int launch_attn(const CUtensorMap& map, dim3 grid, int H, int Nq, float scale, const CaArgs& ca,
                const SaArgs& sa, int32_t* st, cudaStream_t s) {
  const size_t smem = sizeof(AttnSmem) + 1024;
  if (cudaFuncSetAttribute(attn_tc_kernel<kT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_CUDA;
  }
  attn_tc_kernel<kT><<<grid, 128, smem, s>>>(map, H, Nq, scale, ca, sa, st);
  FASTAR_LAUNCHED(s, kT < 0 ? "annca_tc" : "annsa_tc");
  return FASTAR_OK;
}

}  // namespace

size_t annsa_tc_ws_bytes(int H, int Nq, int D, int T) {
  if (D != kD || T > kMaxT) return 0;
  const size_t o = (size_t)T * H * Nq * kD * sizeof(float);
  const size_t ml = (size_t)T * H * Nq * sizeof(float2);
  return ((o + 255) & ~(size_t)255) + ((ml + 255) & ~(size_t)255);
}

int launch_annca_tc(fastar_dtype dt, const void* q, const void* k_p, const void* v_p,
                    const int32_t* kept_idx, const int32_t* kept_cnt, int H, int F, int n_f, int P, int D,
                    float scale, void* out, int32_t* st, cudaStream_t s) {
  if (dt != FASTAR_BF16 || D != kD) return FASTAR_ERR_UNSUPPORTED;
  const int Nq = F * n_f;
  if (Nq == 0 || H == 0) return FASTAR_OK;
  CUtensorMap mapQ;
  if (make_tmap_bf16_2d(&mapQ, q, (uint64_t)H * Nq, kD, kM, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  CaArgs ca{(const __nv_bfloat16*)k_p, (const __nv_bfloat16*)v_p, kept_idx, kept_cnt, F, n_f, P,
            (__nv_bfloat16*)out};
  SaArgs sa{};
  return launch_attn<-1>(mapQ, dim3((n_f + kM - 1) / kM, F, H), H, Nq, scale, ca, sa, st, s);
}

int launch_annsa_tc(fastar_dtype dt, const void* q, const uint32_t* q_codes, const int32_t* q_perm,
                    const int32_t* q_offsets, int Nq, const fastar_cache* c, float scale, void* out,
                    float* lse, void* ws, int32_t* st, cudaStream_t s) {
  (void)q_offsets;
  if (dt != FASTAR_BF16 || c->D != kD || c->T > kMaxT) return FASTAR_ERR_UNSUPPORTED;
  if (Nq == 0 || c->H == 0) return FASTAR_OK;
  if (!ws) return FASTAR_ERR_WORKSPACE;
  const size_t o_bytes = ((size_t)c->T * c->H * Nq * kD * sizeof(float) + 255) & ~(size_t)255;
  SaArgs sa{(const __nv_bfloat16*)q, q_codes, q_perm, (const __nv_bfloat16*)c->K,
            (const __nv_bfloat16*)c->V, c->m, c->codes, c->size, c->perm, c->offsets, c->C, c->T,
            1 << c->B, (float*)ws, (float2*)((char*)ws + o_bytes)};
  CaArgs ca{};
  CUtensorMap dummy;
  memset(&dummy, 0, sizeof(dummy));
  const dim3 grid((Nq + kM - 1) / kM, 1, c->H);
  int rc = FASTAR_OK;
  for (int t = 0; t < c->T && rc == FASTAR_OK; ++t) {
    switch (t) {
      case 0: rc = launch_attn<0>(dummy, grid, c->H, Nq, scale, ca, sa, st, s); break;
      case 1: rc = launch_attn<1>(dummy, grid, c->H, Nq, scale, ca, sa, st, s); break;
      case 2: rc = launch_attn<2>(dummy, grid, c->H, Nq, scale, ca, sa, st, s); break;
      default: rc = launch_attn<3>(dummy, grid, c->H, Nq, scale, ca, sa, st, s); break;
    }
  }
  if (rc != FASTAR_OK) return rc;
  annsa_combine_kernel<<<dim3((Nq + 7) / 8, c->H), 256, 0, s>>>(sa.ws_o, sa.ws_ml, c->T, c->H, Nq,
                                                                 (__nv_bfloat16*)out, lse, st);
  FASTAR_LAUNCHED(s, "annsa_combine");
  return FASTAR_OK;
}

}  // namespace fastar
