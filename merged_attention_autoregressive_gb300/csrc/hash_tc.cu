// Random-hyperplane LSH codes on the tensor cores (tcgen05, bf16).
//
// codes[h][t][i] = sum_b [planes[t*B+b] . x[h][i] > 0] << b
// (FAST-AR summary, paperlayer.ai, section 2 LSH / section 5 ANN attention;
// gist.science technical summary 2.B: one shared LSH space for queries,
// keys and prompt keys; paper.rainbus.top: the hash is computed once and
// serves all three modules.)
//
// The projection is a skinny GEMM: 128 rows of x (K = 128) against the
// T*B hyperplanes (N = T*B rounded up to 16, zero rows past T*B).  The work
// is bound by reading x.  One launch hashes up to kMaxJobs inputs (the
// chunk's queries, new keys and prompt keys), whose 128-row tiles form one
// sequence dealt round-robin to a persistent grid of one CTA per SM.  Each
// CTA keeps a ring of 6 row tiles (32 KiB each) in flight with TMA (two
// 64-column boxes, 128-byte swizzle); one thread issues the 8 MMAs of the
// next tile into the other of two TMEM accumulators before the 4 warps turn
// the signs of the current tile's projections into T codes.  Products are
// exact in fp32 and summed in fp32.
#include <string.h>

#include "common.cuh"
#include "tc.cuh"

namespace fastar {

namespace {

constexpr int kM = 128, kD = 128, kStages = 6, kMaxNP = 64, kMaxJobs = FASTAR_MAX_HASH_JOBS;

struct HashSmem {
  uint8_t X[kStages][kM * kD * 2];
  uint8_t R[kMaxNP * kD * 2];
  uint64_t full[kStages];
  uint64_t mma_done[2];
  uint32_t tmem;
};

struct HashMaps {
  CUtensorMap m[kMaxJobs];
};
struct HashJobs {
  int n;                         // jobs
  int N[kMaxJobs];               // rows per head
  long long rows[kMaxJobs];      // H * N
  int tile0[kMaxJobs + 1];       // first tile of each job in the joint sequence
  uint32_t* codes[kMaxJobs];     // [H][T][N]
};

__device__ __forceinline__ int job_of(const HashJobs& J, int g) {
  int j = 0;
#pragma unroll
  for (int k = 1; k < kMaxJobs; ++k)
    if (k < J.n && g >= J.tile0[k]) j = k;
  return j;
}

__global__ void __launch_bounds__(128, 1) hash_tc_kernel(const __grid_constant__ HashMaps maps,
                                                         const __grid_constant__ HashJobs J,
                                                         const __nv_bfloat16* __restrict__ planes, int TB,
                                                         int NP, int T, int B, int32_t* st) {
  extern __shared__ uint8_t smem_raw[];
  HashSmem& sm = *reinterpret_cast<HashSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5;
  // barriers and TMEM do not depend on the previous kernel; the rows and
  // the hyperplanes may, so they are read after the wait
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) tc::mbar_init(&sm.full[s], 1);
    tc::mbar_init(&sm.mma_done[0], 1);
    tc::mbar_init(&sm.mma_done[1], 1);
    tc::fence_mbar_init();
    for (int j = 0; j < J.n; ++j) tc::prefetch_tensormap(&maps.m[j]);
  }
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem, 128);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;
  pdl_wait();
  if (block_status_bad(st)) {
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
    return;
  }

  // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int ntiles = J.tile0[J.n];
  const int first = blockIdx.x, step = gridDim.x;
  const int mine = first < ntiles ? (ntiles - 1 - first) / step + 1 : 0;
  auto issue = [&](int k, int stage) {
    const int g = first + k * step, j = job_of(J, g);
    const int row0 = (g - J.tile0[j]) * kM;
    tc::mbar_arrive_expect_tx(&sm.full[stage], kM * kD * 2);
    tc::tma_load_2d(sm.X[stage], &maps.m[j], &sm.full[stage], 0, row0);
    tc::tma_load_2d(sm.X[stage] + kM * 128, &maps.m[j], &sm.full[stage], 64, row0);
  };
  if (tid == 0)
    for (int k = 0; k < kStages && k < mine; ++k) issue(k, k);
  // hyperplanes: NP rows, zero past T*B (lands while the first tiles load)
  tc::gather_rows_sw128(tc::smem_u32(sm.R), NP,
                        [&](int r) -> const void* { return r < TB ? (const void*)(planes + (size_t)r * kD) : nullptr; },
                        tid, 128, planes);
  tc::cp_async_commit();
  tc::cp_async_wait_all();
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  const uint32_t idesc = tc::idesc_bf16_f32(kM, NP, 0, 0);
  const uint64_t rdesc = tc::sdesc_kmajor_sw128(tc::smem_u32(sm.R));
  // MMAs of tile k into accumulator k & 1 (one thread)
  auto mma = [&](int k) -> bool {
    const int stage = k % kStages;
    if (!tc::mbar_wait(&sm.full[stage], (uint32_t)(k / kStages) & 1u)) return false;
    tc::tc_fence_after();
    const uint64_t xdesc = tc::sdesc_kmajor_sw128(tc::smem_u32(sm.X[stage]));
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t ox = (kk >> 2) * kM * 128 + (kk & 3) * 32;
      const uint32_t orr = (kk >> 2) * NP * 128 + (kk & 3) * 32;
      tc::mma_bf16(tmem + (uint32_t)((k & 1) * kMaxNP), tc::sdesc_add(xdesc, ox), tc::sdesc_add(rdesc, orr),
                   idesc, kk > 0 ? 1u : 0u);
    }
    tc::mma_commit(&sm.mma_done[k & 1]);
    return true;
  };
  bool ok = true;
  if (tid == 0 && mine > 0) ok = mma(0);
  for (int k = 0; k < mine; ++k) {
    // the next tile's MMAs go into the other accumulator, whose codes were
    // taken before the barrier that ended the previous iteration
    if (tid == 0 && ok && k + 1 < mine) ok = mma(k + 1);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    ok = __all_sync(0xffffffffu, tc::mbar_wait(&sm.mma_done[k & 1], (uint32_t)(k >> 1) & 1u));
    ok = __syncthreads_and(ok);
    if (!ok) break;
    tc::tc_fence_after();
    // the stage is consumed: refill it with the tile kStages ahead
    if (tid == 0 && k + kStages < mine) issue(k + kStages, k % kStages);
    // epilogue: thread = row of the tile
    const uint32_t acc = tmem + (uint32_t)((k & 1) * kMaxNP);
    float v[kMaxNP];
    tc::tmem_ld32(acc + ((uint32_t)(warp * 32) << 16), v);
    if (NP > 32) {
      tc::tmem_ld32(acc + ((uint32_t)(warp * 32) << 16) + 32, v + 32);
    } else {
#pragma unroll
      for (int r = 32; r < kMaxNP; ++r) v[r] = 0.f;
    }
    const int g = first + k * step, j = job_of(J, g);
    const long long row = (long long)(g - J.tile0[j]) * kM + tid;
    if (row < J.rows[j]) {
      // sign bits of the NP projections, bit r = hyperplane r
      unsigned long long bits = 0ull;
#pragma unroll
      for (int r = 0; r < kMaxNP; ++r) bits |= (unsigned long long)(v[r] > 0.f ? 1u : 0u) << r;
      const int N = J.N[j];
      const long long hh = row / N, i = row - hh * N;
      const unsigned long long cmask = (1ull << B) - 1ull;
      uint32_t* codes = J.codes[j];
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

// Up to FASTAR_MAX_HASH_JOBS inputs [H][N_j][D] with one set of hyperplanes.
int launch_hash_tc_many(fastar_dtype dt, int n, const void* const* xs, const int* Ns, uint32_t* const* codes,
                        int H, int D, const void* planes, int T, int B, int32_t* st, cudaStream_t s) {
  if (dt != FASTAR_BF16 || D != kD || T > 8 || T * B > kMaxNP || n < 1 || n > kMaxJobs)
    return FASTAR_ERR_UNSUPPORTED;
  HashMaps maps;
  HashJobs J;
  memset(&maps, 0, sizeof(maps));
  memset(&J, 0, sizeof(J));
  int tiles = 0;
  for (int j = 0; j < n; ++j) {
    const long long rows = (long long)H * Ns[j];
    J.tile0[J.n] = tiles;
    if (rows == 0) continue;
    if (make_tmap_bf16_2d(&maps.m[J.n], xs[j], (uint64_t)rows, kD, kM, 64) != FASTAR_OK) return FASTAR_ERR_CUDA;
    J.N[J.n] = Ns[j];
    J.rows[J.n] = rows;
    J.codes[J.n] = codes[j];
    tiles += (int)((rows + kM - 1) / kM);
    ++J.n;
  }
  J.tile0[J.n] = tiles;
  if (J.n == 0) return FASTAR_OK;
  const int TB = T * B, NP = (TB + 15) / 16 * 16;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  (void)cudaGetLastError();
  const int grid = tiles < sms ? tiles : sms;
  const size_t smem = sizeof(HashSmem) + 1024;
  if (cudaFuncSetAttribute(hash_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_CUDA;
  }
  fastar::launch_pdl((hash_tc_kernel), grid, 128, smem, s, maps, J, (const __nv_bfloat16*)planes, TB, NP, T, B, st);
  FASTAR_LAUNCHED(s, "hash_tc");
  return FASTAR_OK;
}

int launch_hash_tc(fastar_dtype dt, const void* x, int H, int N, int D, const void* planes, int T, int B,
                   uint32_t* codes, int32_t* st, cudaStream_t s) {
  return launch_hash_tc_many(dt, 1, &x, &N, &codes, H, D, planes, T, B, st, s);
}

}  // namespace fastar
