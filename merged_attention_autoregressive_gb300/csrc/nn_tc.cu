// TempCache nearest-neighbour match on the tensor cores (tcgen05, bf16).
//
// For one frame of new keys (FAST-AR summary, paperlayer.ai section 5
// "TempCache": top-1 correspondence; paper.rainbus.top method steps): every
// new key k_j is compared with every candidate group (the groups refreshed in
// the previous frame) by cosine, and matched to the best one (ties: lowest
// slot) iff the cosine reaches tau.
//
// One CTA (4 warps) owns 128 new keys of one head.  The keys arrive by TMA
// (two 64-column boxes, 128-byte swizzle).  Candidate rows are gathered with
// cp.async into the same swizzled layout, 128 at a time, double-buffered so
// the next gather overlaps the current MMA: for the first frame of a call
// they are the cache rows listed by the candidate compaction; for later
// frames they are the previous frame's representative rows of k_new (the
// rows the previous merge step stored into the cache).  One thread issues
// 8 MMAs (M 128, N 128, K 16) into a 128-column fp32 TMEM accumulator; each
// thread then reads its key's 128 dot products from TMEM, scales them by the
// two inverse norms and keeps the best (cosine, slot).
#include <math.h>

#include "common.cuh"
#include "tc.cuh"

namespace fastar {

namespace {

constexpr int kM = 128, kN = 128, kD = 128;
constexpr int kMember = 0;  // plan kind of a key that joined a group it does not represent

struct NnSmem {
  uint8_t A[kM * kD * 2];
  uint8_t B[2][kN * kD * 2];
  float inv_nb[2][kN];
  int slot[2][kN];
  uint64_t bar_a, bar_mma;
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

__global__ void __launch_bounds__(128) nn_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                                                    const __nv_bfloat16* __restrict__ k_new, int n_f,
                                                    int Nrow, int fi, const __nv_bfloat16* __restrict__ K,
                                                    int C, const int32_t* __restrict__ cand,
                                                    const int32_t* __restrict__ ncand,
                                                    const int32_t* __restrict__ prev_slot,
                                                    const int32_t* __restrict__ prev_kind, float tau,
                                                    int32_t* __restrict__ match, int32_t* match_out,
                                                    int32_t* st) {
  extern __shared__ uint8_t smem_raw[];
  NnSmem& sm = *reinterpret_cast<NnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  if (block_status_bad(st)) return;
  const int h = blockIdx.y, m0 = blockIdx.x * kM;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nc = (fi == 0) ? min(max(ncand[h], 0), C) : n_f;
  const int ntiles = (nc + kN - 1) / kN;

  if (tid == 0) {
    tc::mbar_init(&sm.bar_a, 1);
    tc::mbar_init(&sm.bar_mma, 1);
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&mapA);
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem, 128);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;

  if (tid == 0) {
    const int row0 = h * Nrow + fi * n_f + m0;
    tc::mbar_arrive_expect_tx(&sm.bar_a, kM * kD * 2);
    tc::tma_load_2d(sm.A, &mapA, &sm.bar_a, 0, row0);
    tc::tma_load_2d(sm.A + kM * 128, &mapA, &sm.bar_a, 64, row0);
  }

  auto issue_b = [&](int t, int buf) {
    const int c0 = t * kN;
    tc::gather_rows_sw128(
        tc::smem_u32(sm.B[buf]), kN,
        [&](int r) -> const void* {
          const int c = c0 + r;
          if (c >= nc) return nullptr;
          if (fi == 0) return K + ((size_t)h * C + cand[(size_t)h * C + c]) * kD;
          return k_new + ((size_t)h * Nrow + (size_t)(fi - 1) * n_f + c) * kD;
        },
        tid, 128, K);
    tc::cp_async_commit();
    for (int r = tid; r < kN; r += 128) {
      const int c = c0 + r;
      int s = -1;
      if (c < nc) {
        if (fi == 0)
          s = cand[(size_t)h * C + c];
        else
          s = prev_kind[(size_t)h * n_f + c] != kMember ? prev_slot[(size_t)h * n_f + c] : -1;
      }
      sm.slot[buf][r] = s;
    }
  };
  if (ntiles > 0) issue_b(0, 0);

  bool ok = tc::mbar_wait(&sm.bar_a, 0);
  const float na2 = row_sq_norm(sm.A, tid, kM);
  const float ia = na2 > 0.f ? 1.f / sqrtf(na2) : 0.f;
  float best = -INFINITY;
  int best_slot = 0x7fffffff;
  constexpr uint32_t idesc = tc::idesc_bf16_f32(kM, kN, 0, 0);
  uint32_t phase = 0;

  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    tc::cp_async_wait_all();
    tc::fence_proxy_async_smem();
    __syncthreads();
    const float nb2 = row_sq_norm(sm.B[buf], tid, kN);
    sm.inv_nb[buf][tid] = nb2 > 0.f ? 1.f / sqrtf(nb2) : 0.f;
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (tid == 0 && ok) {
      const uint32_t a0 = tc::smem_u32(sm.A), b0 = tc::smem_u32(sm.B[buf]);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off_a = (kk >> 2) * kM * 128 + (kk & 3) * 32;
        const uint32_t off_b = (kk >> 2) * kN * 128 + (kk & 3) * 32;
        tc::mma_bf16(tmem, tc::sdesc_kmajor_sw128(a0 + off_a), tc::sdesc_kmajor_sw128(b0 + off_b), idesc,
                     kk > 0 ? 1u : 0u);
      }
      tc::mma_commit(&sm.bar_mma);
    }
    if (t + 1 < ntiles) issue_b(t + 1, buf ^ 1);
    if (ok) ok = tc::mbar_wait(&sm.bar_mma, phase);
    phase ^= 1;
    tc::tc_fence_after();
    if (ok) {
#pragma unroll 1
      for (int q = 0; q < kN / 32; ++q) {
        float v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + q * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int r = q * 32 + i;
          const int s = sm.slot[buf][r];
          const float ib = sm.inv_nb[buf][r];
          if (s < 0 || ib == 0.f) continue;
          const float cs = v[i] * ia * ib;
          if (cs > best || (cs == best && s < best_slot)) {
            best = cs;
            best_slot = s;
          }
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();
  }
  tc::cp_async_wait_all();
  const int j = m0 + tid;
  if (!ok) {
    if (tid == 0) status_set(st, FASTAR_ERR_TIMEOUT);
  } else if (j < n_f) {
    const int m = (na2 > 0.f && best >= tau) ? best_slot : -1;
    match[(size_t)h * n_f + j] = m;
    if (match_out) match_out[(size_t)h * Nrow + fi * n_f + j] = m;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

}  // namespace

int launch_nn_tc(fastar_dtype dt, const void* k_new, int n_f, int Nrow, int H, int fi, const void* K,
                 int C, int D, const int32_t* cand, const int32_t* ncand, const int32_t* prev_slot,
                 const int32_t* prev_kind, float tau, int32_t* match, int32_t* match_out, int32_t* st,
                 cudaStream_t s) {
  if (dt != FASTAR_BF16 || D != kD) return FASTAR_ERR_UNSUPPORTED;
  if (n_f == 0 || H == 0) return FASTAR_OK;
  CUtensorMap mapA;
  if (make_tmap_bf16_2d(&mapA, k_new, (uint64_t)H * Nrow, kD, kM, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  const size_t smem = sizeof(NnSmem) + 1024;
  if (cudaFuncSetAttribute(nn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_CUDA;
  }
  dim3 grid((n_f + kM - 1) / kM, H);
  nn_tc_kernel<<<grid, 128, smem, s>>>(mapA, (const __nv_bfloat16*)k_new, n_f, Nrow, fi,
                                       (const __nv_bfloat16*)K, C, cand, ncand, prev_slot, prev_kind,
                                       tau, match, match_out, st);
  FASTAR_LAUNCH_CHECK();
  return FASTAR_OK;
}

}  // namespace fastar
