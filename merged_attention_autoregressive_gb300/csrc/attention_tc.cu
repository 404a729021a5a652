// Tensor-core AnnCA / AnnSA attention (tcgen05 + TMEM); bf16 fast path.
#include "common.cuh"

namespace fastar {
int launch_annca_tc(fastar_dtype, const void*, const void*, const void*, const int32_t*,
                    const int32_t*, int, int, int, int, int, float, void*, int32_t*, cudaStream_t) {
  return FASTAR_ERR_UNSUPPORTED;
}
int launch_annsa_tc(fastar_dtype, const void*, const uint32_t*, const int32_t*, const int32_t*, int,
                    const fastar_cache*, float, void*, float*, void*, int32_t*, cudaStream_t) {
  return FASTAR_ERR_UNSUPPORTED;
}
size_t annsa_tc_ws_bytes(int, int, int, int) { return 0; }
}  // namespace fastar
