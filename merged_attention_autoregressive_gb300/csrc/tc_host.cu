// Host helpers of the tensor-core kernels: TMA tensor maps.
//
// The tensor-map encoder is a driver entry point; it is looked up through
// the runtime (cudaGetDriverEntryPointByVersion) on first use, so the library
// does not link the driver library and still loads on a machine without one.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tc.cuh"

namespace fastar {

static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    (void)cudaGetLastError();
  });
  return fn;
}

int make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, uint32_t box_cols) {
  if (((uintptr_t)base & 15) || (cols * 2) % 16 || box_cols * 2 > 128) return FASTAR_ERR_ARG;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const PFN_cuTensorMapEncodeTiled_v12000 encode = encode_tiled_fn();
  if (!encode) return FASTAR_ERR_CUDA;
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                      dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FASTAR_OK : FASTAR_ERR_CUDA;
}

}  // namespace fastar
