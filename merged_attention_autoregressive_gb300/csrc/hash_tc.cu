// Tensor-core LSH projection (tcgen05); filled in by the bf16 fast path.
#include "common.cuh"

namespace fastar {
int launch_hash_tc(fastar_dtype, const void*, int, int, int, const void*, int, int, uint32_t*,
                   int32_t*, cudaStream_t) {
  return FASTAR_ERR_UNSUPPORTED;
}
}  // namespace fastar
