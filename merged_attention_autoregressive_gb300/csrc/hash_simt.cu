// Random-hyperplane LSH codes, one warp per row (CUDA cores).
//
// codes[h][t][i] = sum_b [planes[t*B+b] . x[h][i] > 0] << b
// (FAST-AR summary, paperlayer.ai, section 2 LSH / section 5 ANN attention;
// gist.science technical summary 2.B, one shared LSH space.)
//
// This path serves fp32 inputs; bf16 inputs use the tensor-core kernel in
// hash_tc.cu when it is available for the shape.
#include "common.cuh"

namespace fastar {

template <typename T, int D>
__global__ void __launch_bounds__(256) hash_warp_kernel(const T* __restrict__ x, int rows,
                                                        const T* __restrict__ planes, int T_,
                                                        int B, int N, uint32_t* __restrict__ codes,
                                                        int32_t* st) {
  pdl_wait();
  constexpr int PER = D / 32;
  __shared__ float R[kMaxTB * D];
  const int TB = T_ * B;
  if (block_status_bad(st)) return;
  for (int i = threadIdx.x; i < TB * D; i += blockDim.x) R[i] = Elem<T>::ld(planes + i);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const T* xr = x + (size_t)row * D;
  float xv[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) xv[k] = Elem<T>::ld(xr + lane + 32 * k);
  const int h = row / N, i = row - h * N;
  for (int t = 0; t < T_; ++t) {
    uint32_t code = 0;
    for (int b = 0; b < B; ++b) {
      const float* r = R + (t * B + b) * D;
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < PER; ++k) s = fmaf(xv[k], r[lane + 32 * k], s);
      s = warp_sum(s);
      code |= (s > 0.f ? 1u : 0u) << b;
    }
    if (lane == 0) codes[((size_t)h * T_ + t) * N + i] = code;
  }
  pdl_trigger();
}

int launch_hash_simt(fastar_dtype dt, const void* x, int H, int N, int D, const void* planes,
                     int T, int B, uint32_t* codes, int32_t* st, cudaStream_t s) {
  const int rows = H * N;
  if (rows == 0) return FASTAR_OK;
  dim3 grid((rows + 7) / 8), block(256);
  if (dt == FASTAR_F32 && D == 64)
    fastar::launch_pdl((hash_warp_kernel<float, 64>), grid, block, 0, s, (const float*)x, rows, (const float*)planes, T, B, N, codes, st);
  else if (dt == FASTAR_F32 && D == 128)
    fastar::launch_pdl((hash_warp_kernel<float, 128>), grid, block, 0, s, (const float*)x, rows, (const float*)planes, T, B, N, codes, st);
  else if (dt == FASTAR_BF16 && D == 64)
    fastar::launch_pdl((hash_warp_kernel<__nv_bfloat16, 64>), grid, block, 0, s, (const __nv_bfloat16*)x, rows, (const __nv_bfloat16*)planes, T, B, N, codes, st);
  else if (dt == FASTAR_BF16 && D == 128)
    fastar::launch_pdl((hash_warp_kernel<__nv_bfloat16, 128>), grid, block, 0, s, (const __nv_bfloat16*)x, rows, (const __nv_bfloat16*)planes, T, B, N, codes, st);
  else
    return FASTAR_ERR_UNSUPPORTED;
  FASTAR_LAUNCHED(s, "hash_warp");
  return FASTAR_OK;
}

}  // namespace fastar
