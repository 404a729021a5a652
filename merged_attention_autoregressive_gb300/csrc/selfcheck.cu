// fastar_check_bounded_wait: runs the error path that every tensor-core
// kernel of this library takes when one of its mbarrier waits runs out.
//
// One CTA of two warps: warp 0 allocates a TMEM block, as the tensor-core
// kernels do, and thread 0 waits on an mbarrier that nothing ever arrives
// on, with the same bounded wait (tc::mbar_wait_polls) those kernels use,
// but with the caller's poll count instead of the two-second default.  When
// the wait gives up the kernel records FASTAR_ERR_TIMEOUT in the sticky
// status word, frees its TMEM and returns, so the context stays usable and
// later kernels see the error and write nothing.  No fault, trap or endless
// loop is involved: the wait is bounded and the barrier is never used again.
#include "common.cuh"
#include "tc.cuh"

namespace fastar {

namespace {

constexpr int kCols = 32;

__global__ void __launch_bounds__(64) bounded_wait_kernel(uint32_t polls, int32_t* st) {
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, kCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (threadIdx.x == 0 && !tc::mbar_wait_polls(&bar, 0u, polls)) status_set(st, FASTAR_ERR_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem_base, kCols);
}

}  // namespace

}  // namespace fastar

extern "C" int fastar_check_bounded_wait(int polls, int32_t* dev_status, cudaStream_t stream) {
  if (!dev_status || polls < 1 || polls > FASTAR_CHECK_WAIT_MAX_POLLS) return FASTAR_ERR_ARG;
  fastar::bounded_wait_kernel<<<1, 64, 0, stream>>>((uint32_t)polls, dev_status);
  if (cudaGetLastError() != cudaSuccess) return FASTAR_ERR_CUDA;
  fastar::after_launch(stream, "bounded_wait");
  return FASTAR_OK;
}
