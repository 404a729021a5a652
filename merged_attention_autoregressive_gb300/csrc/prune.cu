// AnnCA pruning: per (head, frame), keep the prompt tokens that share a
// bucket with at least one query of the frame, in ascending order.
//
// gist.science technical summary 2.B (AnnCA mechanism); paper.rainbus.top
// method steps, AnnCA; paperlayer.ai section 5 "AnnCA".  One CTA per
// (frame, head): the frame's query codes set bits of a per-table occupancy
// bitmap (2^B bits per table) in shared memory, then the prompt is scanned
// in order and compacted with a block-wide prefix sum.
#include "common.cuh"

namespace fastar {

constexpr int kPruneThreads = 512;

__global__ void __launch_bounds__(kPruneThreads) prune_kernel(const uint32_t* __restrict__ q_codes,
                                                              const uint32_t* __restrict__ p_codes, int F,
                                                              int n_f, int P, int Tt, int B,
                                                              int32_t* __restrict__ kept_idx,
                                                              int32_t* __restrict__ kept_cnt, int32_t* st) {
  pdl_wait();
  extern __shared__ uint32_t occ[];  // [T][2^B / 32]
  __shared__ int sh[33];
  if (block_status_bad(st)) return;
  const int f = blockIdx.x, h = blockIdx.y;
  const int words = ((1 << B) + 31) >> 5;
  const uint32_t mask = (B >= 32) ? 0xffffffffu : ((1u << B) - 1u);
  const int Nq = F * n_f;
  for (int i = threadIdx.x; i < Tt * words; i += blockDim.x) occ[i] = 0;
  __syncthreads();
  for (int t = 0; t < Tt; ++t) {
    const uint32_t* qc = q_codes + ((size_t)h * Tt + t) * Nq + (size_t)f * n_f;
    for (int i = threadIdx.x; i < n_f; i += blockDim.x) {
      const uint32_t c = qc[i] & mask;
      atomicOr(&occ[t * words + (c >> 5)], 1u << (c & 31));
    }
  }
  __syncthreads();
  int32_t* out = kept_idx + ((size_t)h * F + f) * P;
  int base = 0;
  for (int p0 = 0; p0 < P; p0 += blockDim.x) {
    const int p = p0 + threadIdx.x;
    int keep = 0;
    if (p < P) {
      for (int t = 0; t < Tt && !keep; ++t) {
        const uint32_t c = p_codes[((size_t)h * Tt + t) * P + p] & mask;
        keep = (occ[t * words + (c >> 5)] >> (c & 31)) & 1u;
      }
    }
    int tot;
    const int pos = block_excl_scan(keep, sh, &tot);
    if (keep) out[base + pos] = p;
    base += tot;
  }
  for (int i = base + threadIdx.x; i < P; i += blockDim.x) out[i] = -1;
  if (threadIdx.x == 0) kept_cnt[(size_t)h * F + f] = base;
  pdl_trigger();
}

int launch_prune(const uint32_t* q_codes, const uint32_t* p_codes, int H, int F, int n_f, int P,
                 int T, int B, int32_t* kept_idx, int32_t* kept_cnt, int32_t* st, cudaStream_t s) {
  if (H == 0 || F == 0) return FASTAR_OK;
  const size_t smem = (size_t)T * (((1 << B) + 31) >> 5) * sizeof(uint32_t);
  if (smem > 48 * 1024) return FASTAR_ERR_UNSUPPORTED;
  fastar::launch_pdl((prune_kernel), dim3(F, H), kPruneThreads, smem, s, q_codes, p_codes, F, n_f, P, T, B, kept_idx,
                                                       kept_cnt, st);
  FASTAR_LAUNCHED(s, "prune");
  return FASTAR_OK;
}

}  // namespace fastar
