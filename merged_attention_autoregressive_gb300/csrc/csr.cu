// Bucket CSR: stable counting sort of ids by code, one CTA per group.
//
// perm[g][.] lists ids 0..n-1 grouped by code, ascending id inside a bucket;
// offsets[g][c] = number of ids with code < c.  Used for the chunk's query
// codes (per head and table) and for the live cache codes.  (Buckets of the
// LSH tables: FAST-AR summary, paperlayer.ai, section 2; AnnSA restricts a
// query to keys of its own buckets, gist.science technical summary 2.C.)
//
// Each of W warps (a power of two, up to 32) owns a contiguous segment of
// the ids.
// Pass 1 counts codes per (warp, bucket) in shared memory; pass 2 scans those
// counts in (bucket, warp) order, which makes the placement stable; pass 3
// walks each segment in order, ranking equal codes inside a warp step with
// match_any.
#include "common.cuh"

namespace fastar {

constexpr int kCsrThreads = 1024;  // up to 32 warps

// cnt holds the (warp, bucket) counts bucket-major with a padded row of W+1
// entries per bucket: warp w's lanes, which hit different buckets, land in
// different banks, and the (bucket, warp) scan order is contiguous.
// Codes a warp holds in registers for passes 1 and 3: up to kCsrRegs per
// lane (segments of up to 32 * kCsrRegs ids); longer segments are read
// again from global memory in pass 3.
constexpr int kCsrRegs = 12;

__global__ void __launch_bounds__(kCsrThreads) csr_kernel(const uint32_t* __restrict__ keys, int N,
                                                          const int32_t* __restrict__ n_dev, int n_div,
                                                          int nb, int lgW, int32_t* __restrict__ perm,
                                                          int32_t* __restrict__ offsets, int32_t* st) {
  pdl_wait();
  extern __shared__ int cnt[];  // [nb][W + 1]
  __shared__ int scan_sh[33];
  if (block_status_bad(st)) return;
  const int W = 1 << lgW, SW = W + 1;
  const int g = blockIdx.x;
  int n = N;
  if (n_dev) n = min(max(n_dev[g / n_div], 0), N);
  const uint32_t* kg = keys + (size_t)g * N;
  int32_t* pg = perm + (size_t)g * N;
  int32_t* og = offsets + (size_t)g * (nb + 1);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  for (int i = threadIdx.x; i < nb * SW; i += blockDim.x) cnt[i] = 0;
  const int seg = (n + W - 1) >> lgW;
  const int beg = min(n, warp * seg), end = min(n, beg + seg);
  // the warp's first 32 * kCsrRegs codes, all loads in flight together
  uint32_t reg[kCsrRegs];
#pragma unroll
  for (int r = 0; r < kCsrRegs; ++r) {
    const int i = beg + r * 32 + lane;
    reg[r] = (warp < W && i < end) ? __ldg(kg + i) : 0xffffffffu;
  }
  __syncthreads();
  bool bad = false;
  if (warp < W) {
#pragma unroll
    for (int r = 0; r < kCsrRegs; ++r) {
      const int i = beg + r * 32 + lane;
      if (i >= end) continue;
      const uint32_t c = reg[r];
      if (c >= (uint32_t)nb) { bad = true; continue; }
      atomicAdd(&cnt[c * SW + warp], 1);
    }
    for (int i = beg + 32 * kCsrRegs + lane; i < end; i += 32) {
      const uint32_t c = __ldg(kg + i);
      if (c >= (uint32_t)nb) { bad = true; continue; }
      atomicAdd(&cnt[c * SW + warp], 1);
    }
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) status_set(st, FASTAR_ERR_DEVICE_ARG);
    return;
  }
  // exclusive scan in (bucket, warp) order; thread t owns a contiguous range
  const int total = nb << lgW;
  const int per = (total + blockDim.x - 1) / blockDim.x;
  const int e0 = min(total, (int)threadIdx.x * per), e1 = min(total, e0 + per);
  int sum = 0;
  for (int e = e0; e < e1; ++e) sum += cnt[(e >> lgW) * SW + (e & (W - 1))];
  int run = block_excl_scan(sum, scan_sh, nullptr);
  for (int e = e0; e < e1; ++e) {
    int* p = &cnt[(e >> lgW) * SW + (e & (W - 1))];
    const int v = *p;
    *p = run;
    run += v;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nb; c += blockDim.x) og[c] = cnt[c * SW];  // warp 0 base of bucket c
  if (threadIdx.x == 0) og[nb] = n;
  // stable scatter, 32 ids of the segment at a time in id order
  if (warp < W) {
    auto place = [&](int i, uint32_t c) {
      const bool valid = i < end;
      if (!valid) c = 0xffffffffu;
      const unsigned peers = __match_any_sync(0xffffffffu, c);
      const int rank = __popc(peers & lanemask_lt());
      int pos = 0;
      if (valid) pos = cnt[c * SW + warp] + rank;
      __syncwarp();
      if (valid) {
        pg[pos] = i;
        if (rank == 0) cnt[c * SW + warp] += __popc(peers);
      }
      __syncwarp();
    };
#pragma unroll
    for (int r = 0; r < kCsrRegs; ++r)
      if (beg + r * 32 < end) place(beg + r * 32 + lane, reg[r]);
    for (int base = beg + 32 * kCsrRegs; base < end; base += 32) {
      const int i = base + lane;
      place(i, i < end ? __ldg(kg + i) : 0xffffffffu);
    }
  }
  pdl_trigger();
}

int launch_csr(const uint32_t* keys, int G, int N, const int32_t* n_dev, int n_div, int nb,
               int32_t* perm, int32_t* offsets, int32_t* st, cudaStream_t s) {
  if (G == 0) return FASTAR_OK;
  if (nb > (1 << kMaxCsrBits)) return FASTAR_ERR_UNSUPPORTED;
  // Up to 32 warps per group, each placing its segment 32 ids per step in
  // order: the (bucket, warp) scan grows with the warps but is spread over
  // the same number of threads, while each warp's serial placement shrinks
  // (with 1,024 buckets: 26 us per group with 8 warps).  The (warp, bucket)
  // counts must fit in shared memory.
  int lgW = 5;
  while (lgW > 0 && (size_t)((1 << lgW) + 1) * nb * sizeof(int) > 200 * 1024) --lgW;
  const size_t smem = (size_t)((1 << lgW) + 1) * nb * sizeof(int);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(csr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_CUDA;
  }
  fastar::launch_pdl((csr_kernel), G, 32 << lgW, smem, s, keys, N, n_dev, n_div > 0 ? n_div : 1, nb, lgW, perm,
                     offsets, st);
  FASTAR_LAUNCHED(s, "csr");
  return FASTAR_OK;
}

}  // namespace fastar
