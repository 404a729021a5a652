// fastar_tempcache_merge_noalloc: the TempCache merge without a caller
// workspace, for callers that cannot allocate device memory.
//
// Some callers cannot hand us a workspace: a plugin running inside a host
// application that owns the GPU's memory budget and does not let its
// plugins allocate, or a C/FFI caller that only holds the cache and input
// pointers given to it and has no device allocator of its own.  This entry
// point takes its scratch from a fixed array in the library's own device
// memory instead.  It is the same merge as fastar_tempcache_merge (it calls
// that entry point with the array as the workspace), so results are
// identical.
//
// Costs and limits:
//   * the array is FASTAR_NOALLOC_SCRATCH_BYTES (16 MiB) of device memory,
//     held by every GPU that loads this library until the process exits;
//   * problems whose merge workspace (fastar_workspace_size with
//     FASTAR_OP_MERGE) exceeds it are rejected with FASTAR_ERR_WORKSPACE;
//   * every call shares the one array: calls that overlap on the GPU (on
//     different streams, or from different threads) race on it and must be
//     ordered by the caller;
//   * the array keeps whatever the last call left in it; the merge needs no
//     part of its workspace to start at zero, so nothing is cleared;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first
//     call before any stream capture.
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_merge_scratch[FASTAR_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_merge_scratch on the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in,
// so the kernels must be given this address instead.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return FASTAR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FASTAR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_merge_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return FASTAR_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FASTAR_OK;
}

}  // namespace

extern "C" int fastar_tempcache_merge_noalloc(const fastar_cache* cache, const void* k_new,
                                              const void* v_new, const uint32_t* codes_new, int F,
                                              int n_f, int32_t first_frame, float tau,
                                              int32_t* match_out, int32_t* dev_status,
                                              cudaStream_t stream) {
  // Argument checks, the no-op cases and the workspace check are the
  // workspace merge's own: the array is handed over only when the call will
  // launch work and the array is large enough; otherwise the merge is given
  // no workspace and answers exactly as fastar_tempcache_merge would (OK for
  // an empty call, ERR_ARG / ERR_UNSUPPORTED for bad arguments, and
  // FASTAR_ERR_WORKSPACE when the problem needs more than the array).
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  if (cache && F > 0 && n_f > 0 && cache->H > 0 && n_f <= cache->C && n_f <= FASTAR_MAX_FRAME_KEYS) {
    const size_t need = fastar_workspace_size(FASTAR_OP_MERGE, cache->H, n_f, cache->D, cache->T,
                                              cache->B, cache->C);
    if (need <= (size_t)FASTAR_NOALLOC_SCRATCH_BYTES) {
      const int rc = scratch_address(&scratch);
      if (rc != FASTAR_OK) return rc;
      scratch_bytes = (size_t)FASTAR_NOALLOC_SCRATCH_BYTES;
    }
  }
  return fastar_tempcache_merge(cache, k_new, v_new, codes_new, F, n_f, first_frame, tau,
                                match_out, scratch, scratch_bytes,
                                dev_status, stream);
}
