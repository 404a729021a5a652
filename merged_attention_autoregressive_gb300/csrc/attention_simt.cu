// AnnCA and AnnSA attention on CUDA cores, one warp per query.
//
// AnnCA (gist.science technical summary 2.B): query i of frame f attends
// the kept prompt tokens of (head, f):  o = sum softmax(scale q.k) v.
// AnnSA (gist.science 2.C, paper.rainbus.top method steps; + ln m from
// paperlayer.ai appendix A, Lemma A.1): query i attends the live cache
// slots sharing a code with it in some table; each table walks its own
// bucket of the cache CSR and skips slots an earlier table already
// admitted, so every allowed slot is visited exactly once.
// Online softmax in fp32 (running max, rescaled sum and accumulator).
// This path serves fp32 inputs; bf16 inputs use the tensor-core kernels.
#include <math.h>

#include "common.cuh"

namespace fastar {

template <int PER>
struct OnlineSoftmax {
  float mx = -INFINITY, l = 0.f, acc[PER];
  __device__ OnlineSoftmax() {
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  }
  template <typename T>
  __device__ __forceinline__ void add(float s, const T* vrow, int lane) {
    const float mn = fmaxf(mx, s);
    const float corr = __expf(mx - mn);  // mx = -inf on the first key: 0
    const float p = __expf(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = fmaf(p, Elem<T>::ld(vrow + lane + 32 * i), acc[i] * corr);
    mx = mn;
  }
};

template <typename T, int D>
__global__ void __launch_bounds__(256) annca_simt_kernel(const T* __restrict__ q, const T* __restrict__ k_p,
                                                         const T* __restrict__ v_p,
                                                         const int32_t* __restrict__ kept_idx,
                                                         const int32_t* __restrict__ kept_cnt, int F, int n_f,
                                                         int P, float scale, T* __restrict__ out,
                                                         int32_t* st) {
  pdl_wait();
  constexpr int PER = D / 32;
  if (status_bad(st)) return;
  const int h = blockIdx.y;
  const int Nq = F * n_f;
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= Nq) return;
  const int f = i / n_f;
  const T* qr = q + ((size_t)h * Nq + i) * D;
  float qv[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) qv[k] = Elem<T>::ld(qr + lane + 32 * k) * scale;
  const int cnt = min(max(kept_cnt[(size_t)h * F + f], 0), P);
  const int32_t* ids = kept_idx + ((size_t)h * F + f) * P;
  OnlineSoftmax<PER> os;
  bool bad = false;
  for (int c = 0; c < cnt; ++c) {
    const int p = ids[c];
    if (p < 0 || p >= P) { bad = true; continue; }
    const T* kr = k_p + ((size_t)h * P + p) * D;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) s = fmaf(qv[k], Elem<T>::ld(kr + lane + 32 * k), s);
    s = warp_sum(s);
    os.add(s, v_p + ((size_t)h * P + p) * D, lane);
  }
  if (bad && lane == 0) status_set(st, FASTAR_ERR_DEVICE_ARG);
  const float inv = os.l > 0.f ? 1.f / os.l : 0.f;
  T* orow = out + ((size_t)h * Nq + i) * D;
#pragma unroll
  for (int k = 0; k < PER; ++k) Elem<T>::st(orow + lane + 32 * k, os.acc[k] * inv);
  pdl_trigger();
}

template <typename T, int D>
__global__ void __launch_bounds__(256) annsa_simt_kernel(const T* __restrict__ q, const uint32_t* __restrict__ q_codes,
                                                         int Nq, const T* __restrict__ K, const T* __restrict__ V,
                                                         const int32_t* __restrict__ m,
                                                         const uint32_t* __restrict__ codes,
                                                         const int32_t* __restrict__ size,
                                                         const int32_t* __restrict__ perm,
                                                         const int32_t* __restrict__ offsets, int C, int Tt,
                                                         int nb, float scale, T* __restrict__ out,
                                                         float* __restrict__ lse, int32_t* st) {
  pdl_wait();
  constexpr int PER = D / 32;
  if (status_bad(st)) return;
  const int h = blockIdx.y;
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= Nq) return;
  const T* qr = q + ((size_t)h * Nq + i) * D;
  float qv[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) qv[k] = Elem<T>::ld(qr + lane + 32 * k) * scale;
  uint32_t qc[8];
  for (int t = 0; t < Tt; ++t) qc[t] = q_codes[((size_t)h * Tt + t) * Nq + i];
  const int n = min(max(size[h], 0), C);
  OnlineSoftmax<PER> os;
  for (int t = 0; t < Tt; ++t) {
    const uint32_t c = qc[t];
    if (c >= (uint32_t)nb) continue;
    const int32_t* off = offsets + ((size_t)h * Tt + t) * (nb + 1);
    const int b0 = max(off[c], 0), b1 = min(off[c + 1], n);
    const int32_t* pp = perm + ((size_t)h * Tt + t) * C;
    for (int e = b0; e < b1; ++e) {
      const int s = pp[e];
      if (s < 0 || s >= n) continue;
      bool dup = false;
      for (int u = 0; u < t; ++u) dup |= codes[((size_t)h * Tt + u) * C + s] == qc[u];
      if (dup) continue;
      const T* kr = K + ((size_t)h * C + s) * D;
      float dot = 0.f;
#pragma unroll
      for (int k = 0; k < PER; ++k) dot = fmaf(qv[k], Elem<T>::ld(kr + lane + 32 * k), dot);
      dot = warp_sum(dot);
      const float sc = dot + logf((float)m[(size_t)h * C + s]);
      os.add(sc, V + ((size_t)h * C + s) * D, lane);
    }
  }
  const float inv = os.l > 0.f ? 1.f / os.l : 0.f;
  T* orow = out + ((size_t)h * Nq + i) * D;
#pragma unroll
  for (int k = 0; k < PER; ++k) Elem<T>::st(orow + lane + 32 * k, os.acc[k] * inv);
  if (lse && lane == 0) lse[(size_t)h * Nq + i] = os.l > 0.f ? os.mx + logf(os.l) : -INFINITY;
  pdl_trigger();
}

int launch_annca_simt(fastar_dtype dt, const void* q, const void* k_p, const void* v_p,
                      const int32_t* kept_idx, const int32_t* kept_cnt, int H, int F, int n_f, int P,
                      int D, float scale, void* out, int32_t* st, cudaStream_t s) {
  const int Nq = F * n_f;
  if (Nq == 0 || H == 0) return FASTAR_OK;
  dim3 grid((Nq + 7) / 8, H), block(256);
#define ANNCA_CASE(TT, DD)                                                                      \
  fastar::launch_pdl((annca_simt_kernel<TT, DD>), grid, block, 0, s, (const TT*)q, (const TT*)k_p, (const TT*)v_p, \
                                                   kept_idx, kept_cnt, F, n_f, P, scale, (TT*)out, st)
  if (dt == FASTAR_F32 && D == 64) ANNCA_CASE(float, 64);
  else if (dt == FASTAR_F32 && D == 128) ANNCA_CASE(float, 128);
  else if (dt == FASTAR_BF16 && D == 64) ANNCA_CASE(__nv_bfloat16, 64);
  else if (dt == FASTAR_BF16 && D == 128) ANNCA_CASE(__nv_bfloat16, 128);
  else return FASTAR_ERR_UNSUPPORTED;
#undef ANNCA_CASE
  FASTAR_LAUNCHED(s, "annca_simt");
  return FASTAR_OK;
}

int launch_annsa_simt(fastar_dtype dt, const void* q, const uint32_t* q_codes, int Nq,
                      const fastar_cache* c, float scale, void* out, float* lse, int32_t* st,
                      cudaStream_t s) {
  if (Nq == 0 || c->H == 0) return FASTAR_OK;
  dim3 grid((Nq + 7) / 8, c->H), block(256);
  const int nb = 1 << c->B;
#define ANNSA_CASE(TT, DD)                                                                        \
  fastar::launch_pdl((annsa_simt_kernel<TT, DD>), grid, block, 0, s, (const TT*)q, q_codes, Nq, (const TT*)c->K,    \
                                                   (const TT*)c->V, c->m, c->codes, c->size,      \
                                                   c->perm, c->offsets, c->C, c->T, nb, scale,    \
                                                   (TT*)out, lse, st)
  if (dt == FASTAR_F32 && c->D == 64) ANNSA_CASE(float, 64);
  else if (dt == FASTAR_F32 && c->D == 128) ANNSA_CASE(float, 128);
  else if (dt == FASTAR_BF16 && c->D == 64) ANNSA_CASE(__nv_bfloat16, 64);
  else if (dt == FASTAR_BF16 && c->D == 128) ANNSA_CASE(__nv_bfloat16, 128);
  else return FASTAR_ERR_UNSUPPORTED;
#undef ANNSA_CASE
  FASTAR_LAUNCHED(s, "annsa_simt");
  return FASTAR_OK;
}

}  // namespace fastar
