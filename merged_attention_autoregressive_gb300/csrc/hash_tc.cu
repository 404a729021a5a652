// Random-hyperplane LSH codes on the tensor cores (tcgen05, bf16).
//
// codes[h][t][i] = sum_b [planes[t*B+b] . x[h][i] > 0] << b
// (FAST-AR summary, paperlayer.ai, section 2 LSH / section 5 ANN attention;
// gist.science technical summary 2.B: one shared LSH space for queries,
// keys and prompt keys.)
//
// The projection is a skinny GEMM: 128 rows of x (K = 128) against the
// T*B hyperplanes (N = T*B rounded up to 16, zero rows past T*B).  The work
// is bound by reading x, so the kernel is persistent: each CTA keeps a ring
// of 4 row tiles (32 KiB each) in flight with TMA (two 64-column boxes,
// 128-byte swizzle), one thread issues the 8 MMAs of a tile into one of two
// TMEM accumulators, and the 4 warps turn the signs of their row's N
// projections into T codes.  Products are exact in fp32 and summed in fp32.
#include "common.cuh"
#include "tc.cuh"

namespace fastar {

namespace {

constexpr int kM = 128, kD = 128, kStages = 4, kMaxNP = 64;

struct HashSmem {
  uint8_t X[kStages][kM * kD * 2];
  uint8_t R[kMaxNP * kD * 2];
  uint64_t full[kStages];
  uint64_t mma_done[2];
  uint32_t tmem;
};

__global__ void __launch_bounds__(128, 1) hash_tc_kernel(const __grid_constant__ CUtensorMap mapX,
                                                         const __nv_bfloat16* __restrict__ planes, int TB,
                                                         int NP, int T, int B, int N, long long rows, int ntiles,
                                                         uint32_t* __restrict__ codes, int32_t* st) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  HashSmem& sm = *reinterpret_cast<HashSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  if (block_status_bad(st)) return;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) tc::mbar_init(&sm.full[s], 1);
    tc::mbar_init(&sm.mma_done[0], 1);
    tc::mbar_init(&sm.mma_done[1], 1);
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&mapX);
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem, 128);
    tc::tmem_relinquish();
  }
  // hyperplanes: NP rows, zero past T*B
  tc::gather_rows_sw128(tc::smem_u32(sm.R), NP,
                        [&](int r) -> const void* { return r < TB ? (const void*)(planes + (size_t)r * kD) : nullptr; },
                        tid, 128, planes);
  tc::cp_async_commit();
  tc::cp_async_wait_all();
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;

  // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int first = blockIdx.x, step = gridDim.x;
  const int mine = first < ntiles ? (ntiles - 1 - first) / step + 1 : 0;
  if (tid == 0) {
    for (int k = 0; k < kStages && k < mine; ++k) {
      const int tile = first + k * step;
      tc::mbar_arrive_expect_tx(&sm.full[k], kM * kD * 2);
      tc::tma_load_2d(sm.X[k], &mapX, &sm.full[k], 0, tile * kM);
      tc::tma_load_2d(sm.X[k] + kM * 128, &mapX, &sm.full[k], 64, tile * kM);
    }
  }
  const uint32_t idesc = tc::idesc_bf16_f32(kM, NP, 0, 0);
  bool ok = true;
  for (int k = 0; k < mine && ok; ++k) {
    const int stage = k % kStages, buf = k & 1;
    const uint32_t full_phase = (uint32_t)(k / kStages) & 1u;
    const uint32_t mma_phase = (uint32_t)(k >> 1) & 1u;
    const uint32_t acc = tmem + (uint32_t)(buf * kMaxNP);
    if (tid == 0) {
      ok = tc::mbar_wait(&sm.full[stage], full_phase);
      if (ok) {
        tc::tc_fence_after();
        const uint32_t x0 = tc::smem_u32(sm.X[stage]), r0 = tc::smem_u32(sm.R);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t ox = (kk >> 2) * kM * 128 + (kk & 3) * 32;
          const uint32_t orr = (kk >> 2) * NP * 128 + (kk & 3) * 32;
          tc::mma_bf16(acc, tc::sdesc_kmajor_sw128(x0 + ox), tc::sdesc_kmajor_sw128(r0 + orr), idesc,
                       kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sm.mma_done[buf]);
      }
    }
    ok = __syncthreads_and(ok);
    if (!ok) break;
    ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.mma_done[buf], mma_phase));
    ok = __syncthreads_and(ok);
    if (!ok) break;
    tc::tc_fence_after();
    // the stage is consumed: refill it with the tile kStages ahead
    if (tid == 0 && k + kStages < mine) {
      const int tile = first + (k + kStages) * step;
      tc::mbar_arrive_expect_tx(&sm.full[stage], kM * kD * 2);
      tc::tma_load_2d(sm.X[stage], &mapX, &sm.full[stage], 0, tile * kM);
      tc::tma_load_2d(sm.X[stage] + kM * 128, &mapX, &sm.full[stage], 64, tile * kM);
    }
    // epilogue: thread = row of the tile
    float v[kMaxNP];
    tc::tmem_ld32(acc + ((uint32_t)(warp * 32) << 16), v);
    if (NP > 32) {
      tc::tmem_ld32(acc + ((uint32_t)(warp * 32) << 16) + 32, v + 32);
    } else {
#pragma unroll
      for (int r = 32; r < kMaxNP; ++r) v[r] = 0.f;
    }
    const long long row = (long long)(first + k * step) * kM + tid;
    if (row < rows) {
      // sign bits of the NP projections, bit r = hyperplane r
      unsigned long long bits = 0ull;
#pragma unroll
      for (int r = 0; r < kMaxNP; ++r) bits |= (unsigned long long)(v[r] > 0.f ? 1u : 0u) << r;
      const long long hh = row / N, i = row - hh * N;
      const unsigned long long cmask = (1ull << B) - 1ull;
      for (int t = 0; t < T; ++t) codes[(hh * T + t) * N + i] = (uint32_t)((bits >> (t * B)) & cmask);
    }
    tc::tc_fence_before();
    __syncthreads();
  }
  if (!ok && tid == 0) status_set(st, FASTAR_ERR_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
  pdl_trigger();
}

}  // namespace

int launch_hash_tc(fastar_dtype dt, const void* x, int H, int N, int D, const void* planes, int T, int B,
                   uint32_t* codes, int32_t* st, cudaStream_t s) {
  if (dt != FASTAR_BF16 || D != kD || T > 8 || T * B > kMaxNP) return FASTAR_ERR_UNSUPPORTED;
  const long long rows = (long long)H * N;
  if (rows == 0) return FASTAR_OK;
  CUtensorMap mapX;
  if (make_tmap_bf16_2d(&mapX, x, (uint64_t)rows, kD, kM, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
  const int TB = T * B, NP = (TB + 15) / 16 * 16;
  const int ntiles = (int)((rows + kM - 1) / kM);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  (void)cudaGetLastError();
  const int grid = ntiles < sms ? ntiles : sms;
  const size_t smem = sizeof(HashSmem) + 1024;
  if (cudaFuncSetAttribute(hash_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_CUDA;
  }
  fastar::launch_pdl((hash_tc_kernel), grid, 128, smem, s, mapX, (const __nv_bfloat16*)planes, TB, NP, T, B, N, rows, ntiles,
                                         codes, st);
  FASTAR_LAUNCHED(s, "hash_tc");
  return FASTAR_OK;
}

}  // namespace fastar
