// The quantised matcher on the GPU (FAST-AR summary, paperlayer.ai, section 5
// "ANN Attention": keep the keys of largest query-key product, found by LSH
// or by quantised similarity search without offline preprocessing, and
// appendix C "Quantization precision for ANN matching": 2 to 32 bits;
// paper.rainbus.top, reproduction: FAISS, 8-bit codes by default).
//
// Per head, the searched vectors (live cache keys, prompt keys, or a
// TempCache frame's candidates) get a per-dimension uniform quantiser over
// their own range [lo, hi]:
//   code = floor((x - lo) / (hi - lo) * (2^b - 1) + 0.5), clipped to [0, 2^b - 1]
//   (0 where hi == lo), computed in fp64 with correctly rounded operations in
//   exactly that order, so that the integer codes are those of the plain
//   fp64 definition; decoded vector lo + code (hi - lo) / (2^b - 1), in fp32.
// AnnSA-Quant / AnnCA-Quant: every query keeps the k keys of largest
// approximate score scale q . decoded + bias (ties: lower index) and attends
// them exactly: the attention kernel runs over every key with a per-query
// selection mask.  TempCache-Quant: each new key takes the candidate of
// largest approximate cosine (ties: lowest slot) and merges iff the exact
// cosine of that candidate reaches tau (the plan decides on it).
//
// Kernels: a two-stage per-dimension range, the encoder (warp per row), a
// 64 x 64-tiled fp32 score kernel on the CUDA cores (decoded keys staged in
// shared memory; scores written out, or reduced to each row's best
// approximate cosine), and a per-row radix select that writes the mask.
#include <math.h>

#include <algorithm>

#include "common.cuh"

namespace fastar {

namespace {

constexpr int kD = 128;
constexpr int kRangeBlocks = 16;
constexpr int kTile = 64, kKc = 32;      // score tile: 64 rows x 64 keys, 32 dims per step
constexpr size_t kScoreBytes = 1ull << 30;  // scores kept at once (heads are batched to fit)

// The rows of one head that are searched: position c < count(h) is row
// idx[h * idx_stride + c] (or c) of x[h * rows_per_head + row][D].
struct RowSet {
  const __nv_bfloat16* x;
  long long rows_per_head;
  const int32_t* idx;
  int idx_stride;
  const int32_t* n_dev;  // per-head count (nullable: n_cap)
  int n_cap;
};
__device__ __forceinline__ int rs_count(const RowSet& rs, int h, bool* over) {
  const int n = rs.n_dev ? rs.n_dev[h] : rs.n_cap;
  if (n > rs.n_cap && over) *over = true;
  return min(max(n, 0), rs.n_cap);
}
__device__ __forceinline__ int rs_row(const RowSet& rs, int h, int c) {
  return rs.idx ? rs.idx[(size_t)h * rs.idx_stride + c] : c;
}

// Partial per-dimension minimum and maximum: grid (kRangeBlocks, H), one
// thread per dimension.
__global__ void __launch_bounds__(kD) sq_range_partial_kernel(RowSet rs, float* part, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  const int h = blockIdx.y, d = threadIdx.x;
  bool over = false;
  const int n = rs_count(rs, h, &over);
  float lo = INFINITY, hi = -INFINITY;
  bool bad = false;
#pragma unroll 4
  for (int c = blockIdx.x; c < n; c += gridDim.x) {
    const int r = rs_row(rs, h, c);
    if (r < 0 || r >= rs.rows_per_head) {
      bad = true;
      continue;
    }
    const float v = __bfloat162float(rs.x[((size_t)h * rs.rows_per_head + r) * kD + d]);
    lo = fminf(lo, v);
    hi = fmaxf(hi, v);
  }
  float* p = part + ((size_t)h * kRangeBlocks + blockIdx.x) * 2 * kD;
  p[d] = lo;
  p[kD + d] = hi;
  if ((bad || over) && d == 0) status_set(st, FASTAR_ERR_DEVICE_ARG);
  pdl_trigger();
}

// lohi[h][0][d] = lo, lohi[h][1][d] = hi: grid H, one thread per dimension.
__global__ void __launch_bounds__(kD) sq_range_final_kernel(const float* part, float* lohi, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  const int h = blockIdx.x, d = threadIdx.x;
  float lo = INFINITY, hi = -INFINITY;
  for (int b = 0; b < kRangeBlocks; ++b) {
    const float* p = part + ((size_t)h * kRangeBlocks + b) * 2 * kD;
    lo = fminf(lo, p[d]);
    hi = fmaxf(hi, p[kD + d]);
  }
  lohi[(size_t)h * 2 * kD + d] = lo;
  lohi[(size_t)h * 2 * kD + kD + d] = hi;
  pdl_trigger();
}

// fp64 code of x: the operations of the definition, each correctly rounded
// and none fused.
__device__ __forceinline__ uint32_t sq_code(double x, double lo, double hi, double L) {
  const double span = __dsub_rn(hi, lo);
  const double u = span > 0.0 ? __ddiv_rn(__dsub_rn(x, lo), span) : 0.0;
  double c = floor(__dadd_rn(__dmul_rn(u, L), 0.5));
  c = fmin(fmax(c, 0.0), L);
  return (uint32_t)c;
}

// Codes [H][n_cap][D] of the rows (warp per row, 4 dimensions per lane) and,
// when dec_inv is given, the inverse norm of each decoded row (NaN for a
// zero row).  grid (ceil(n_cap / 8), H), 256 threads.
template <typename CodeT>
__global__ void __launch_bounds__(256) sq_encode_kernel(RowSet rs, const float* lohi, int bits, CodeT* codes,
                                                        float* dec_inv, int ld_inv, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  const int h = blockIdx.y, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int n = rs_count(rs, h, nullptr);
  if (c >= n) return;
  const int r = rs_row(rs, h, c);
  if (r < 0 || r >= rs.rows_per_head) return;  // reported by the range kernel
  const double L = (double)((1u << bits) - 1u);
  const float* lo = lohi + (size_t)h * 2 * kD;
  const float* hi = lo + kD;
  const uint2 raw = *reinterpret_cast<const uint2*>(rs.x + ((size_t)h * rs.rows_per_head + r) * kD + lane * 4);
  const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(&raw);
  uint32_t cd[4];
  float n2 = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int d = lane * 4 + e;
    cd[e] = sq_code((double)__bfloat162float(xv[e]), (double)lo[d], (double)hi[d], L);
    const float step = (hi[d] - lo[d]) / (float)L;
    const float dec = fmaf((float)cd[e], step, lo[d]);
    n2 = fmaf(dec, dec, n2);
  }
  CodeT* out = codes + ((size_t)h * rs.n_cap + c) * kD + lane * 4;
#pragma unroll
  for (int e = 0; e < 4; ++e) out[e] = (CodeT)cd[e];
  n2 = warp_sum(n2);
  if (dec_inv && lane == 0) dec_inv[(size_t)h * ld_inv + c] = n2 > 0.f ? 1.f / sqrtf(n2) : __int_as_float(0x7fc00000);
  pdl_trigger();
}

struct ScoreArgs {
  const __nv_bfloat16* a;  // rows [H][a_rows][D]: queries or new keys
  long long a_rows;
  int Na;                  // rows used per head
  const void* codes;       // [H][n_cap][D]
  int n_cap;
  const int32_t* n_dev;    // per-head key count (nullable: n_cap)
  const float* lohi;       // [H][2][D]
  int bits;
  float scale;
  // scores mode
  const int32_t* m;        // bias ln m[h * m_stride + c] (nullable: 0)
  int m_stride;
  float* scores;           // [hb][Na][n_cap] for heads h0 .. h0 + hb - 1
  int h0;
  // best-cosine mode
  const float* dec_inv;    // [H][ld_inv]
  int ld_inv;
  const int32_t* cand;     // slots of the candidates [H][cand_stride]
  int cand_stride;
  const __nv_bfloat16* K;  // cache keys [H][C][D]
  int C;
  unsigned long long* best;  // [H][Na]
};

// 64 rows x 64 keys of dot products a . decoded key (fp32, K in steps of 32
// dimensions through shared memory); thread (ty, tx) owns rows 4 ty .. 4 ty
// + 3 and keys 4 tx .. 4 tx + 3.
template <typename CodeT>
__device__ __forceinline__ void score_tile(const ScoreArgs& p, int h, int r0, int c0, int nkeys,
                                           float (&As)[kKc][kTile + 4], float (&Bs)[kKc][kTile + 4],
                                           const float* s_lo, const float* s_step, float (&acc)[4][4]) {
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const CodeT* codes = reinterpret_cast<const CodeT*>(p.codes);
  const int lr = tid >> 2, lch = (tid & 3) * 8;  // loader: row / key lr, dims lch .. lch + 7 of the step
  for (int d0 = 0; d0 < kD; d0 += kKc) {
    {
      const int i = r0 + lr;
      float av[8];
      if (i < p.Na) {
        const uint4 raw = *reinterpret_cast<const uint4*>(p.a + ((size_t)h * p.a_rows + i) * kD + d0 + lch);
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
        for (int k = 0; k < 8; ++k) av[k] = __bfloat162float(e[k]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) av[k] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) As[lch + k][lr] = av[k];
      const int c = c0 + lr;
      float bv[8];
      if (c < nkeys) {
        const CodeT* src = codes + ((size_t)h * p.n_cap + c) * kD + d0 + lch;
#pragma unroll
        for (int k = 0; k < 8; ++k) bv[k] = fmaf((float)src[k], s_step[d0 + lch + k], s_lo[d0 + lch + k]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) bv[k] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) Bs[lch + k][lr] = bv[k];
    }
    __syncthreads();
#pragma unroll 8
    for (int dd = 0; dd < kKc; ++dd) {
      const float4 a4 = *reinterpret_cast<const float4*>(&As[dd][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4*>(&Bs[dd][tx * 4]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void load_quantiser(const ScoreArgs& p, int h, float* s_lo, float* s_step) {
  for (int d = threadIdx.x; d < kD; d += blockDim.x) {
    const float lo = p.lohi[(size_t)h * 2 * kD + d], hi = p.lohi[(size_t)h * 2 * kD + kD + d];
    s_lo[d] = lo;
    s_step[d] = (hi - lo) / (float)((1u << p.bits) - 1u);
  }
}

// Scores of heads h0 .. h0 + gridDim.z - 1: grid (key tiles, row tiles, hb).
template <typename CodeT>
__global__ void __launch_bounds__(256) quant_scores_kernel(ScoreArgs p, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  __shared__ __align__(16) float As[kKc][kTile + 4];
  __shared__ __align__(16) float Bs[kKc][kTile + 4];
  __shared__ float s_lo[kD], s_step[kD];
  const int hh = blockIdx.z, h = p.h0 + hh;
  const int nkeys = p.n_dev ? min(max(p.n_dev[h], 0), p.n_cap) : p.n_cap;
  const int c0 = blockIdx.x * kTile, r0 = blockIdx.y * kTile;
  if (c0 >= nkeys || r0 >= p.Na) return;
  load_quantiser(p, h, s_lo, s_step);
  __syncthreads();
  float acc[4][4];
  score_tile<CodeT>(p, h, r0, c0, nkeys, As, Bs, s_lo, s_step, acc);
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  float bias[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = c0 + tx * 4 + j;
    bias[j] = (p.m && c < nkeys) ? logf((float)max(p.m[(size_t)h * p.m_stride + c], 1)) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= p.Na) continue;
    float* out = p.scores + ((size_t)hh * p.Na + r) * p.n_cap + c0 + tx * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (c0 + tx * 4 + j < nkeys) out[j] = fmaf(p.scale, acc[i][j], bias[j]);
  }
  pdl_trigger();
}

// TempCache-Quant: per new key, the candidate of largest approximate cosine
// (dot with the decoded candidate times its inverse decoded norm; ties to
// the lowest slot), then that candidate's exact cosine, packed with its slot
// for the plan (0: no candidate).  grid (1, row tiles, H).
template <typename CodeT>
__global__ void __launch_bounds__(256) quant_best_kernel(ScoreArgs p, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  __shared__ __align__(16) float As[kKc][kTile + 4];
  __shared__ __align__(16) float Bs[kKc][kTile + 4];
  __shared__ float s_lo[kD], s_step[kD];
  __shared__ float s_inv[kTile];
  __shared__ int s_slot[kTile];
  __shared__ int s_best[kTile];
  const int h = blockIdx.z;
  const int nkeys = p.n_dev ? min(max(p.n_dev[h], 0), p.n_cap) : p.n_cap;
  const int r0 = blockIdx.y * kTile;
  if (r0 >= p.Na) return;
  load_quantiser(p, h, s_lo, s_step);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float best[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  int bslot[4] = {0x7fffffff, 0x7fffffff, 0x7fffffff, 0x7fffffff};
  int bpos[4] = {-1, -1, -1, -1};
  for (int c0 = 0; c0 < nkeys; c0 += kTile) {
    __syncthreads();  // the previous tile's s_inv / s_slot are read
    if (tid < kTile) {
      const int c = c0 + tid;
      s_inv[tid] = c < nkeys ? p.dec_inv[(size_t)h * p.ld_inv + c] : __int_as_float(0x7fc00000);
      s_slot[tid] = c < nkeys ? p.cand[(size_t)h * p.cand_stride + c] : 0x7fffffff;
    }
    float acc[4][4];
    score_tile<CodeT>(p, h, r0, c0, nkeys, As, Bs, s_lo, s_step, acc);  // its barriers publish s_inv
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = tx * 4 + j;
        const float v = acc[i][j] * s_inv[col];  // NaN (no candidate, zero norm) never wins
        const int sl = s_slot[col];
        if (v > best[i] || (v == best[i] && sl < bslot[i])) {
          best[i] = v;
          bslot[i] = sl;
          bpos[i] = c0 + col;
        }
      }
    }
  }
  // the 16 threads of a row group (one half-warp) hold candidates of the
  // same rows: keep the best (lowest slot on ties)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best[i], o);
      const int os = __shfl_xor_sync(0xffffffffu, bslot[i], o);
      const int op = __shfl_xor_sync(0xffffffffu, bpos[i], o);
      if (ov > best[i] || (ov == best[i] && os < bslot[i])) {
        best[i] = ov;
        bslot[i] = os;
        bpos[i] = op;
      }
    }
    if (tx == 0) s_best[ty * 4 + i] = bpos[i] >= 0 ? bslot[i] : -1;
  }
  __syncthreads();
  // exact cosine of each row's chosen candidate: a warp per row
  const int warp = tid >> 5, lane = tid & 31;
  bool bad = false;
  for (int rr = warp; rr < kTile; rr += 8) {
    const int i = r0 + rr;
    if (i >= p.Na) break;
    const int sl = s_best[rr];
    unsigned long long out = 0ull;
    if (sl >= 0 && sl < p.C) {
      const uint2 ka = *reinterpret_cast<const uint2*>(p.a + ((size_t)h * p.a_rows + i) * kD + lane * 4);
      const uint2 kb = *reinterpret_cast<const uint2*>(p.K + ((size_t)h * p.C + sl) * kD + lane * 4);
      const __nv_bfloat16* ea = reinterpret_cast<const __nv_bfloat16*>(&ka);
      const __nv_bfloat16* eb = reinterpret_cast<const __nv_bfloat16*>(&kb);
      float dot = 0.f, na = 0.f, nb = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = __bfloat162float(ea[e]), y = __bfloat162float(eb[e]);
        dot = fmaf(x, y, dot);
        na = fmaf(x, x, na);
        nb = fmaf(y, y, nb);
      }
      dot = warp_sum(dot);
      na = warp_sum(na);
      nb = warp_sum(nb);
      if (na > 0.f && nb > 0.f) out = pack_best(dot / (sqrtf(na) * sqrtf(nb)), sl);
    } else if (sl >= p.C) {
      bad = true;
    }
    if (lane == 0) p.best[(size_t)h * p.Na + i] = out;
  }
  if (bad && lane == 0) status_set(st, FASTAR_ERR_DEVICE_ARG);
  pdl_trigger();
}

// The selection mask of one row: the k_eff = min(k, n) positions of largest
// score, ties to the lower position; mask[(hh * Na + i) * words + w] bit b
// is position 32 w + b.  A radix select (11, 11, 10 bits of the scores'
// order-preserving integer keys) finds the k-th largest key T; then the
// positions with key > T and the first (k_eff - #{key > T}) with key == T
// are set.  grid (Na, hb), 256 threads.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(__fadd_rn(v, 0.f));  // -0 and +0 are one value
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(256) topk_mask_kernel(const float* scores, int Na, int n_cap, const int32_t* n_dev,
                                                        int h0, int k, uint32_t* mask, int words, int32_t* st) {
  pdl_wait();
  if (status_bad(st)) return;
  __shared__ int hist[2048];
  __shared__ int sh[33];
  __shared__ uint32_t s_prefix, s_pmask;
  __shared__ int s_need;
  const int i = blockIdx.x, hh = blockIdx.y, h = h0 + hh;
  const int n = n_dev ? min(max(n_dev[h], 0), n_cap) : n_cap;
  const float* row = scores + ((size_t)hh * Na + i) * n_cap;
  uint32_t* mrow = mask + ((size_t)h * Na + i) * words;
  const int tid = threadIdx.x;
  const int keff = min(max(k, 0), n);
  if (keff == n || keff == 0) {
    for (int w = tid; w < words; w += blockDim.x) {
      const int lo = w * 32;
      uint32_t bits = 0u;
      if (keff > 0 && lo < n) bits = (n - lo >= 32) ? 0xffffffffu : ((1u << (n - lo)) - 1u);
      mrow[w] = bits;
    }
    pdl_trigger();
    return;
  }
  if (tid == 0) {
    s_prefix = 0u;
    s_pmask = 0u;
    s_need = keff;
  }
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int nbin = 1 << widths[pass], sh_b = shifts[pass];
    for (int b = tid; b < nbin; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, pmask = s_pmask;
    for (int c = tid; c < n; c += blockDim.x) {
      const uint32_t u = order_key(row[c]);
      if ((u & pmask) == prefix) atomicAdd(&hist[(u >> sh_b) & (nbin - 1)], 1);
    }
    __syncthreads();
    // bins from the top: thread t sums bins [nbin - (t+1) per, nbin - t per)
    const int per = nbin / 256;
    int sum = 0;
    for (int q = 0; q < per; ++q) sum += hist[nbin - 1 - (tid * per + q)];
    int tot;
    const int before = block_excl_scan(sum, sh, &tot);  // count in higher bins than this thread's
    const int need = s_need;
    if (before < need && before + sum >= need) {
      int cum = before;
      for (int q = 0; q < per; ++q) {
        const int b = nbin - 1 - (tid * per + q);
        if (cum + hist[b] >= need) {
          s_prefix = prefix | ((uint32_t)b << sh_b);
          s_pmask = pmask | ((uint32_t)(nbin - 1) << sh_b);
          s_need = need - cum;
          break;
        }
        cum += hist[b];
      }
    }
    __syncthreads();
  }
  const uint32_t T = s_prefix;
  const int need_eq = s_need;  // positions with key == T to keep, lowest first
  // emit in chunks of blockDim.x consecutive positions (one mask word per warp)
  int eq_base = 0;
  const int lane = tid & 31, warp = tid >> 5;
  for (int c0 = 0; c0 < words * 32; c0 += blockDim.x) {
    const int c = c0 + tid;
    uint32_t u = 0u;
    const bool in = c < n;
    if (in) u = order_key(row[c]);
    const int is_eq = (in && u == T) ? 1 : 0;
    int eq_tot;
    const int eq_before = block_excl_scan(is_eq, sh, &eq_tot) + eq_base;
    const bool sel = in && (u > T || (is_eq && eq_before < need_eq));
    const uint32_t bits = __ballot_sync(0xffffffffu, sel);
    const int w = (c0 >> 5) + warp;
    if (lane == 0 && w < words) mrow[w] = bits;
    eq_base += eq_tot;
  }
  pdl_trigger();
}

// The one-bucket description of a key set for the attention kernel: every
// query and every key in bucket 0 of a single table, in index order, so that
// the kernel walks all keys of the head and the selection mask decides.
__global__ void __launch_bounds__(256) onebucket_kernel(int H, int Nq, int N, const int32_t* n_dev, uint32_t* qc,
                                                        int32_t* qp, int32_t* q_off, uint32_t* cc, int32_t* cp,
                                                        int32_t* c_off, int32_t* ones, int32_t* size_out) {
  pdl_wait();
  const size_t tq = (size_t)H * Nq, tc = (size_t)H * N;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < tq + tc; e += (size_t)gridDim.x * blockDim.x) {
    if (e < tq) {
      qc[e] = 0u;
      qp[e] = (int32_t)(e % Nq);
    } else {
      const size_t f = e - tq;
      cc[f] = 0u;
      cp[f] = (int32_t)(f % N);
      if (ones) ones[f] = 1;
    }
  }
  if (blockIdx.x == 0) {
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
      const int n = n_dev ? min(max(n_dev[h], 0), N) : N;
      q_off[h * 3 + 0] = 0;
      q_off[h * 3 + 1] = Nq;
      q_off[h * 3 + 2] = Nq;
      c_off[h * 3 + 0] = 0;
      c_off[h * 3 + 1] = n;
      c_off[h * 3 + 2] = n;
      if (size_out) size_out[h] = N;
    }
  }
  pdl_trigger();
}

inline size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

struct QuantWs {
  float* part;
  float* lohi;
  void* codes;
  float* scores;
  uint32_t* mask;
  uint32_t* qc;
  int32_t* qp;
  int32_t* q_off;
  uint32_t* cc;
  int32_t* cp;
  int32_t* c_off;
  int32_t* ones;
  int32_t* size;
  int hb, words;
};

int heads_per_batch(int H, int Nq, int N) {
  const size_t per = (size_t)Nq * (size_t)N * sizeof(float);
  size_t hb = per ? kScoreBytes / per : (size_t)H;
  if (hb < 1) hb = 1;
  if (hb > (size_t)H) hb = H;
  return (int)hb;
}

size_t quant_ws_layout(int H, int Nq, int N, int bits, void* base, QuantWs* w) {
  const int hb = heads_per_batch(H, Nq, N);
  const int words = (N + 31) / 32;
  const size_t code_b = bits <= 8 ? 1 : 2;
  size_t off = 0;
  char* p = (char*)base;
  auto take = [&](size_t bytes) { void* r = p ? (void*)(p + off) : nullptr; off += a256(bytes); return r; };
  QuantWs ws;
  ws.part = (float*)take((size_t)H * kRangeBlocks * 2 * kD * 4);
  ws.lohi = (float*)take((size_t)H * 2 * kD * 4);
  ws.codes = take((size_t)H * N * kD * code_b);
  ws.scores = (float*)take((size_t)hb * Nq * N * 4);
  ws.mask = (uint32_t*)take((size_t)H * Nq * words * 4);
  ws.qc = (uint32_t*)take((size_t)H * Nq * 4);
  ws.qp = (int32_t*)take((size_t)H * Nq * 4);
  ws.q_off = (int32_t*)take((size_t)H * 3 * 4);
  ws.cc = (uint32_t*)take((size_t)H * N * 4);
  ws.cp = (int32_t*)take((size_t)H * N * 4);
  ws.c_off = (int32_t*)take((size_t)H * 3 * 4);
  ws.ones = (int32_t*)take((size_t)H * N * 4);
  ws.size = (int32_t*)take((size_t)H * 4);
  ws.hb = hb;
  ws.words = words;
  if (w) *w = ws;
  return off;
}

template <typename CodeT>
int run_range_encode(const RowSet& rs, int H, int bits, float* part, float* lohi, CodeT* codes, float* dec_inv,
                     int ld_inv, int32_t* st, cudaStream_t s) {
  fastar::launch_pdl((sq_range_partial_kernel), dim3(kRangeBlocks, H), kD, 0, s, rs, part, st);
  FASTAR_LAUNCHED(s, "sq_range");
  fastar::launch_pdl((sq_range_final_kernel), dim3(H), kD, 0, s, (const float*)part, lohi, st);
  FASTAR_LAUNCHED(s, "sq_range_final");
  fastar::launch_pdl((sq_encode_kernel<CodeT>), dim3((rs.n_cap + 7) / 8, H), 256, 0, s, rs, (const float*)lohi, bits,
                     codes, dec_inv, ld_inv, st);
  FASTAR_LAUNCHED(s, "sq_encode");
  return FASTAR_OK;
}

// The keys of `c` (K, V, m, size; C keys per head) attended by each query of
// q with the k keys of largest approximate score kept: range, codes, scores
// and selection per head batch, then the attention kernel over every key
// with the selection mask.
template <typename CodeT>
int quant_attend(const void* q, int Nq, const fastar_cache* c, const int32_t* m_for_bias, float scale, int topk,
                 int bits, void* out, float* lse, uint32_t* sel_mask, const QuantWs& w, int32_t* st, cudaStream_t s) {
  const int H = c->H, N = c->C;
  RowSet rs{(const __nv_bfloat16*)c->K, N, nullptr, 0, c->size, N};
  int rc = run_range_encode<CodeT>(rs, H, bits, w.part, w.lohi, (CodeT*)w.codes, nullptr, 0, st, s);
  if (rc != FASTAR_OK) return rc;
  uint32_t* mask = sel_mask ? sel_mask : w.mask;
  for (int h0 = 0; h0 < H; h0 += w.hb) {
    const int hb = std::min(w.hb, H - h0);
    ScoreArgs p{};
    p.a = (const __nv_bfloat16*)q;
    p.a_rows = Nq;
    p.Na = Nq;
    p.codes = w.codes;
    p.n_cap = N;
    p.n_dev = c->size;
    p.lohi = w.lohi;
    p.bits = bits;
    p.scale = scale;
    p.m = m_for_bias;
    p.m_stride = N;
    p.scores = w.scores;
    p.h0 = h0;
    fastar::launch_pdl((quant_scores_kernel<CodeT>), dim3((N + kTile - 1) / kTile, (Nq + kTile - 1) / kTile, hb), 256,
                       0, s, p, st);
    FASTAR_LAUNCHED(s, "quant_scores");
    fastar::launch_pdl((topk_mask_kernel), dim3(Nq, hb), 256, 0, s, (const float*)w.scores, Nq, N, c->size, h0, topk,
                       mask, w.words, st);
    FASTAR_LAUNCHED(s, "topk_mask");
  }
  fastar_cache view = *c;
  view.T = 1;
  view.B = 1;
  view.codes = w.cc;
  view.perm = w.cp;
  view.offsets = w.c_off;
  return launch_annsa_masked(FASTAR_BF16, q, w.qc, w.qp, w.q_off, Nq, &view, scale, out, lse, mask, w.words, st, s);
}

}  // namespace

size_t quant_ws_bytes(int H, int Nq, int N, int D, int bits) {
  if (D != kD || bits < 1 || bits > 16 || H <= 0 || Nq <= 0 || N <= 0) return 0;
  return quant_ws_layout(H, Nq, N, bits, nullptr, nullptr);
}

int launch_annsa_quant(const void* q, int Nq, const fastar_cache* c, float scale, int topk, int bits, void* out,
                       float* lse, uint32_t* sel_mask, void* ws, int32_t* st, cudaStream_t s) {
  QuantWs w;
  quant_ws_layout(c->H, Nq, c->C, bits, ws, &w);
  fastar::launch_pdl((onebucket_kernel), dim3(2 * 148), 256, 0, s, c->H, Nq, c->C, (const int32_t*)c->size, w.qc,
                     w.qp, w.q_off, w.cc, w.cp, w.c_off, (int32_t*)nullptr, (int32_t*)nullptr);
  FASTAR_LAUNCHED(s, "onebucket");
  if (bits <= 8)
    return quant_attend<uint8_t>(q, Nq, c, c->m, scale, topk, bits, out, lse, sel_mask, w, st, s);
  return quant_attend<uint16_t>(q, Nq, c, c->m, scale, topk, bits, out, lse, sel_mask, w, st, s);
}

int launch_annca_quant(const void* q, const void* k_p, const void* v_p, int H, int Nq, int P, float scale, int topk,
                       int bits, void* out, uint32_t* sel_mask, void* ws, int32_t* st, cudaStream_t s) {
  QuantWs w;
  quant_ws_layout(H, Nq, P, bits, ws, &w);
  fastar::launch_pdl((onebucket_kernel), dim3(2 * 148), 256, 0, s, H, Nq, P, (const int32_t*)nullptr, w.qc, w.qp,
                     w.q_off, w.cc, w.cp, w.c_off, w.ones, w.size);
  FASTAR_LAUNCHED(s, "onebucket");
  fastar_cache c{};
  c.H = H;
  c.D = kD;
  c.C = P;
  c.T = 1;
  c.B = 1;
  c.dt = FASTAR_BF16;
  c.K = const_cast<void*>(k_p);
  c.V = const_cast<void*>(v_p);
  c.m = w.ones;
  c.size = w.size;
  // the prompt tokens have no multiplicity: no bias
  if (bits <= 8)
    return quant_attend<uint8_t>(q, Nq, &c, nullptr, scale, topk, bits, out, nullptr, sel_mask, w, st, s);
  return quant_attend<uint16_t>(q, Nq, &c, nullptr, scale, topk, bits, out, nullptr, sel_mask, w, st, s);
}

size_t quant_nn_ws_bytes(int H, int n_f) {
  return a256((size_t)H * kRangeBlocks * 2 * kD * 4) + a256((size_t)H * 2 * kD * 4);
}

// TempCache-Quant for one frame: the candidates cand[h][c < ncand[h]]
// (slots of the cache, at most n_f) are quantised over their own range;
// each of the frame's keys gets its best approximate candidate and that
// candidate's exact cosine in best[h][j].  codes: [H][n_f][D] (2 bytes per
// code), dec_inv: [H][ld_inv].
int launch_quant_nn(const void* k_frame, long long a_rows, int n_f, int H, const void* K, int C, const int32_t* cand,
                    const int32_t* ncand, int bits, void* ws_small, void* codes, float* dec_inv, int ld_inv,
                    unsigned long long* best, int32_t* st, cudaStream_t s) {
  float* part = (float*)ws_small;
  float* lohi = (float*)((char*)ws_small + a256((size_t)H * kRangeBlocks * 2 * kD * 4));
  RowSet rs{(const __nv_bfloat16*)K, C, cand, C, ncand, n_f};
  ScoreArgs p{};
  p.a = (const __nv_bfloat16*)k_frame;
  p.a_rows = a_rows;
  p.Na = n_f;
  p.codes = codes;
  p.n_cap = n_f;
  p.n_dev = ncand;
  p.lohi = lohi;
  p.bits = bits;
  p.dec_inv = dec_inv;
  p.ld_inv = ld_inv;
  p.cand = cand;
  p.cand_stride = C;
  p.K = (const __nv_bfloat16*)K;
  p.C = C;
  p.best = best;
  const dim3 grid(1, (n_f + kTile - 1) / kTile, H);
  if (bits <= 8) {
    int rc = run_range_encode<uint8_t>(rs, H, bits, part, lohi, (uint8_t*)codes, dec_inv, ld_inv, st, s);
    if (rc != FASTAR_OK) return rc;
    fastar::launch_pdl((quant_best_kernel<uint8_t>), grid, 256, 0, s, p, st);
  } else {
    int rc = run_range_encode<uint16_t>(rs, H, bits, part, lohi, (uint16_t*)codes, dec_inv, ld_inv, st, s);
    if (rc != FASTAR_OK) return rc;
    fastar::launch_pdl((quant_best_kernel<uint16_t>), grid, 256, 0, s, p, st);
  }
  FASTAR_LAUNCHED(s, "quant_best");
  return FASTAR_OK;
}

}  // namespace fastar
