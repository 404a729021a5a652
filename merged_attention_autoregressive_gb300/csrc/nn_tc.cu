// Tensor-core TempCache nearest-neighbour match (tcgen05); bf16 fast path.
#include "common.cuh"

namespace fastar {
int launch_nn_tc(fastar_dtype, const void*, int, int, int, const void*, int, int, const int32_t*,
                 const int32_t*, float, int32_t*, int32_t*, int, int32_t*, cudaStream_t) {
  return FASTAR_ERR_UNSUPPORTED;
}
}  // namespace fastar
