// Shared device helpers of the FAST-AR kernels: element access for bf16/fp32,
// the sticky device status word, warp/block scans.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "fastar.h"

namespace fastar {

constexpr int kMaxTB = 64;      // T*B hyperplanes per hash call
constexpr int kMaxCsrBits = 12; // bucket CSR supports up to 4096 buckets

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float ld(const float* p) { return *p; }
  static __device__ __forceinline__ void st(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float ld(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
  }
  static __device__ __forceinline__ void st(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
  }
};

// N consecutive elements of a row moved as one vector (the address is
// aligned to N * sizeof(T), which must be 4, 8 or 16 bytes): raw loads and
// stores, and conversion to / from floats.
template <typename T, int N>
struct VecOf {
  static constexpr int B = N * (int)sizeof(T);
  static_assert(B == 4 || B == 8 || B == 16, "vector width");
  using type = typename std::conditional<B == 4, uint32_t, typename std::conditional<B == 8, uint2, uint4>::type>::type;
};
template <typename T, int N>
__device__ __forceinline__ typename VecOf<T, N>::type ld_raw(const T* p) {
  return *reinterpret_cast<const typename VecOf<T, N>::type*>(p);
}
template <typename T, int N>
__device__ __forceinline__ void st_raw(T* p, const typename VecOf<T, N>::type& v) {
  *reinterpret_cast<typename VecOf<T, N>::type*>(p) = v;
}
template <typename T, int N>
__device__ __forceinline__ void raw_to_float(const typename VecOf<T, N>::type& v, float* out) {
  const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
  for (int i = 0; i < N; ++i) out[i] = Elem<T>::ld(e + i);
}
template <typename T, int N>
__device__ __forceinline__ void ld_vec(const T* p, float* out) {
  raw_to_float<T, N>(ld_raw<T, N>(p), out);
}
template <typename T, int N>
__device__ __forceinline__ void st_vec(T* p, const float* in) {
  typename VecOf<T, N>::type v;
  T* e = reinterpret_cast<T*>(&v);
#pragma unroll
  for (int i = 0; i < N; ++i) Elem<T>::st(e + i, in[i]);
  st_raw<T, N>(p, v);
}

// ---- sticky device status: first error wins, kernels exit once it is set
__device__ __forceinline__ bool status_bad(const int32_t* st) {
  return st != nullptr && *((volatile const int32_t*)st) != 0;
}
__device__ __forceinline__ void status_set(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}
// Block-uniform status check: thread 0 reads the word, every thread gets the
// same answer (a block never splits at a later barrier).  Call from all threads.
__device__ __forceinline__ bool block_status_bad(const int32_t* st) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = status_bad(st) ? 1 : 0;
  __syncthreads();
  const bool bad = s_bad != 0;
  __syncthreads();
  return bad;
}

// A nearest-neighbour candidate (cosine, slot) packed into one 64-bit word
// whose unsigned order is: larger cosine first, then lower slot.  The best
// candidate of several partial searches is their atomicMax; 0 means none.
__device__ __forceinline__ unsigned long long pack_best(float cos, int slot) {
  uint32_t b = __float_as_uint(cos);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)b << 32) | (unsigned long long)(0xffffffffu - (uint32_t)slot);
}
__device__ __forceinline__ float best_cos(unsigned long long key) {
  const uint32_t b = (uint32_t)(key >> 32);
  return __uint_as_float((b & 0x80000000u) ? (b & 0x7fffffffu) : ~b);
}
__device__ __forceinline__ int best_slot(unsigned long long key) {
  return (int)(0xffffffffu - (uint32_t)key);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Exclusive scan over the block (blockDim.x a multiple of 32, <= 1024).
// `sh` holds at least 33 ints.  Returns the exclusive prefix; *total gets
// the block sum.  Every thread must call it.
__device__ __forceinline__ int block_excl_scan(int v, int* sh, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int inc = warp_incl_scan(v);
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sh[lane] : 0;
    int wi = warp_incl_scan(w);
    if (lane < nw) sh[lane] = wi - w;
    if (lane == nw - 1) sh[32] = wi;
  }
  __syncthreads();
  int res = sh[warp] + inc - v;
  if (total) *total = sh[32];
  __syncthreads();
  return res;
}

__device__ __forceinline__ int block_min_int(int v, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sh[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = min(w, __shfl_xor_sync(0xffffffffu, w, o));
    if (lane == 0) sh[32] = w;
  }
  __syncthreads();
  int r = sh[32];
  __syncthreads();
  return r;
}

__device__ __forceinline__ long long block_sum_ll(long long v, long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (lane == 0) sh[32] = w;
  }
  __syncthreads();
  long long r = sh[32];
  __syncthreads();
  return r;
}

}  // namespace fastar

// ---- host-side launch helpers (declared here, defined per .cu file)
namespace fastar {
int launch_hash(fastar_dtype dt, const void* x, int H, int N, int D, const void* planes,
                int T, int B, uint32_t* codes, int32_t* st, cudaStream_t s);
int launch_csr(const uint32_t* keys, int G, int N, const int32_t* n_dev, int n_div, int nb,
               int32_t* perm, int32_t* offsets, int32_t* st, cudaStream_t s);
int launch_merge(const fastar_cache* c, const void* k_new, const void* v_new,
                 const uint32_t* codes_new, int F, int n_f, int32_t first_frame, float tau,
                 int32_t* match_out, void* ws, int32_t* st, cudaStream_t s,
                 cudaEvent_t codes_ready = nullptr, int rep = 0, const void* planes = nullptr,
                 int search = 0);
size_t merge_ws_bytes(int H, int n_f, int C);
int launch_prune(const uint32_t* q_codes, const uint32_t* p_codes, int H, int F, int n_f,
                 int P, int T, int B, int32_t* kept_idx, int32_t* kept_cnt, int32_t* st,
                 cudaStream_t s);
int launch_annca(fastar_dtype dt, const void* q, const void* k_p, const void* v_p,
                 const int32_t* kept_idx, const int32_t* kept_cnt, int H, int F, int n_f,
                 int P, int D, float scale, void* out, void* ws, size_t ws_bytes, int32_t* st, cudaStream_t s);
int launch_annsa(fastar_dtype dt, const void* q, const uint32_t* q_codes,
                 const int32_t* q_perm, const int32_t* q_offsets, int Nq,
                 const fastar_cache* c, float scale, void* out, float* lse, void* ws,
                 int32_t* st, cudaStream_t s);
size_t annsa_ws_bytes(int H, int Nq, int D, int T);
int launch_annsa_masked(fastar_dtype dt, const void* q, const uint32_t* q_codes, const int32_t* q_perm,
                        const int32_t* q_offsets, int Nq, const fastar_cache* c, float scale, void* out, float* lse,
                        const uint32_t* mask, int mask_words, int32_t* st, cudaStream_t s);
size_t quant_ws_bytes(int H, int Nq, int N, int D, int bits);
int launch_annsa_quant(const void* q, int Nq, const fastar_cache* c, float scale, int topk, int bits, void* out,
                       float* lse, uint32_t* sel_mask, void* ws, int32_t* st, cudaStream_t s);
int launch_annca_quant(const void* q, const void* k_p, const void* v_p, int H, int Nq, int P, float scale, int topk,
                       int bits, void* out, uint32_t* sel_mask, void* ws, int32_t* st, cudaStream_t s);
}  // namespace fastar

namespace fastar {
// Called after every kernel launch of the library: counts it and, while
// launch timing is on (fastar_timing_begin), records the next caller event
// on the launch stream, tagged with the kernel's name.
void after_launch(cudaStream_t s, const char* name);

// Every kernel of the library is a programmatic dependent launch: it may be
// scheduled while the previous kernel of the stream is still finishing, so
// its launch and CTA ramp-up overlap that kernel's tail.  Each kernel starts
// with pdl_wait(), which returns once the previous grid has completed and its
// writes are visible (so it must come before any other access, TMEM
// allocation included), and calls pdl_trigger() when its main work is done:
// the next grid is launched once every CTA of this one has triggered or
// exited, so its waiting CTAs only share the SMs with this grid's last ones.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
}

#define FASTAR_LAUNCHED(stream, name)                           \
  do {                                                          \
    fastar::after_launch((stream), (name));                     \
    if (cudaPeekAtLastError() != cudaSuccess) {                 \
      (void)cudaGetLastError();                                 \
      return FASTAR_ERR_CUDA;                                   \
    }                                                           \
  } while (0)
