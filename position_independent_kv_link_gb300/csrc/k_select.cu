// Dynamic (attention-based) choice of the prompt tokens a link recomputes: the CacheBlend-r
// step the EPIC pages measure LegoLink's static choice against (EPIC summary page: problem
// statement; Measured effects table, CacheBlend-r rows and the static-vs-dynamic row). Reading
// of the step: with the prompt linked as compiled (nothing recomputed), the query rows at layer
// 0 attend causally over the prompt and the query, RoPE at absolute positions; a prompt token's
// score is the sum of the softmax weights it receives over all query rows and heads; the
// floor(r N / 100) best-scoring tokens are recomputed (equal scores: the lower position first).
//
// Three kernels per pass, all requests at once, fp32 arithmetic:
//   sel_rowstats_kernel  one warp per (query row, head): rotated, scaled q and the row's softmax
//                        maximum and sum over every key it sees;
//   sel_scores_kernel    one warp per prompt token: its score, summed over heads and query rows
//                        in a fixed order (the same bits on every run);
//   sel_top_kernel       one CTA per request: the n-th largest score found by bisection over the
//                        scores' bit patterns, then a compaction in position order.
#include <cmath>

#include "pic_internal.h"

namespace pic {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTopThreads = 1024;

template <typename T>
__device__ __forceinline__ float kv_f(const T* p) { return to_f<T>(*p); }

// Dims lane + 32 j (j < D/32) of a head vector, rotated at position p: rotate-half pairs
// (i, i + D/2) turn by p theta_i, (cos, sin) from the table row [D/2] of position p.
template <int D>
__device__ __forceinline__ void rotate(const float (&x)[D / 32], int p, const float2* __restrict__ tab,
                                       float (&out)[D / 32]) {
  constexpr int NJ = D / 32;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < NJ / 2; ++j) {
    const float2 c = tab[(size_t)p * (D / 2) + lane + 32 * j];
    const float a = x[j], b = x[j + NJ / 2];
    out[j] = a * c.x - b * c.y;
    out[j + NJ / 2] = b * c.x + a * c.y;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The request whose range [first(i), first(i + 1)) holds x (requests in ascending order).
template <typename F>
__device__ __forceinline__ int find_req(int n_reqs, int x, F first) {
  int lo = 0, hi = n_reqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (first(mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename T, int D>
__global__ void __launch_bounds__(128) sel_rowstats_kernel(SelectArgs a) {
  constexpr int NJ = D / 32;
  const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= a.n_rows * a.H) return;
  const int row = w / a.H, h = w % a.H, g = h / (a.H / a.G);
  const SelectReq& R = a.reqs[find_req(a.n_reqs, row, [&](int i) { return a.reqs[i].row0; })];
  const int s = row - R.row0;
  const int QKV = (a.H + 2 * a.G) * D;
  float x[NJ], q[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) x[j] = a.qkv[(size_t)row * QKV + h * D + lane + 32 * j];
  rotate<D>(x, R.n_tok + s, a.rope_cs, q);
  const float sc = rsqrtf((float)D) * kLog2e;   // scores in log2 units
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    q[j] *= sc;
    a.qrot[((size_t)row * a.H + h) * D + lane + 32 * j] = q[j];
  }
  float m = -INFINITY, l = 0.f;
  auto take = [&](const float (&kx)[NJ], int p) {
    float kr[NJ];
    rotate<D>(kx, p, a.rope_cs, kr);
    float d = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) d += q[j] * kr[j];
    d = warp_sum(d);
    const float mn = fmaxf(m, d);
    l = l * exp2f(m - mn) + exp2f(d - mn);
    m = mn;
  };
  const T* K = static_cast<const T*>(a.k_layer0);
  for (int p = R.page0; p < R.page0 + R.n_pages; ++p) {
    const int blk = a.page_block[p], base = a.page_pos[p], len = a.page_len[p];
    for (int r = 0; r < len; ++r) {
      float kx[NJ];
      const T* kr = K + (((size_t)blk * a.G + g) * kBlock + r) * D;
#pragma unroll
      for (int j = 0; j < NJ; ++j) kx[j] = kv_f<T>(kr + lane + 32 * j);
      take(kx, base + r);
    }
  }
  for (int u = 0; u <= s; ++u) {   // the query's own keys (its layer-0 projections)
    float kx[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) kx[j] = a.qkv[(size_t)(R.row0 + u) * QKV + (a.H + g) * D + lane + 32 * j];
    take(kx, R.n_tok + u);
  }
  if (lane == 0) {
    a.ml[((size_t)row * a.H + h) * 2] = m;
    a.ml[((size_t)row * a.H + h) * 2 + 1] = l;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(128) sel_scores_kernel(SelectArgs a) {
  constexpr int NJ = D / 32;
  const int u_all = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (u_all >= a.n_tok) return;
  const SelectReq& R = a.reqs[find_req(a.n_reqs, u_all, [&](int i) { return a.reqs[i].tok0; })];
  const int u = u_all - R.tok0;
  // the token's page: pages cover the prompt contiguously, in position order
  int lo = R.page0, hi = R.page0 + R.n_pages - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.page_pos[mid] <= u) lo = mid; else hi = mid - 1;
  }
  const int blk = a.page_block[lo], r = u - a.page_pos[lo];
  const T* K = static_cast<const T*>(a.k_layer0);
  const int rep = a.H / a.G;
  float total = 0.f;
  for (int g = 0; g < a.G; ++g) {
    float kx[NJ], kr[NJ];
    const T* kp = K + (((size_t)blk * a.G + g) * kBlock + r) * D;
#pragma unroll
    for (int j = 0; j < NJ; ++j) kx[j] = kv_f<T>(kp + lane + 32 * j);
    rotate<D>(kx, u, a.rope_cs, kr);
    for (int h = g * rep; h < (g + 1) * rep; ++h)
      for (int s = 0; s < R.lq; ++s) {
        const size_t qh = (size_t)(R.row0 + s) * a.H + h;
        const float* q = a.qrot + qh * D;
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < NJ; ++j) d += q[lane + 32 * j] * kr[j];
        d = warp_sum(d);
        total += exp2f(d - a.ml[qh * 2]) / a.ml[qh * 2 + 1];
      }
  }
  if (lane == 0) a.scores[u_all] = total;
}

// Block-wide sum of one int per thread (kTopThreads threads).
__device__ __forceinline__ int block_sum(int v, int* red) {
  v = __reduce_add_sync(0xffffffffu, v);
  __syncthreads();   // earlier readers of red are done
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = 0;
#pragma unroll 8
  for (int i = 0; i < kTopThreads / 32; ++i) t += red[i];
  return t;
}

// Exclusive prefix (over the warps before this one) and total of one int per warp.
__device__ __forceinline__ int2 warp_scan(int per_warp, int* buf) {
  const int wid = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) buf[wid] = per_warp;
  __syncthreads();
  int pre = 0, tot = 0;
  for (int k = 0; k < kTopThreads / 32; ++k) {
    const int c = buf[k];
    pre += k < wid ? c : 0;
    tot += c;
  }
  return make_int2(pre, tot);
}

__global__ void __launch_bounds__(kTopThreads) sel_top_kernel(SelectArgs a) {
  __shared__ int red[kTopThreads / 32];
  const SelectReq& R = a.reqs[blockIdx.x];
  const int N = R.n_tok, n = R.n_pick;
  const uint32_t* bits = reinterpret_cast<const uint32_t*>(a.scores + R.tok0);
  int* out = a.chosen + R.out0;
  if (n <= 0) return;
  // Scores are >= 0, so their bit patterns order like the scores. thr: the largest pattern
  // with at least n scores at or above it -- the n-th largest score.
  uint32_t thr = 0;
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = thr | (1u << b);
    int c = 0;
    for (int i = threadIdx.x; i < N; i += kTopThreads) c += bits[i] >= cand;
    if (block_sum(c, red) >= n) thr = cand;
  }
  int c = 0;
  for (int i = threadIdx.x; i < N; i += kTopThreads) c += bits[i] > thr;
  int eq_left = n - block_sum(c, red);   // scores equal to thr that are kept: the first ones
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
  int base = 0;
  for (int i0 = 0; i0 < N; i0 += kTopThreads) {
    const int i = i0 + threadIdx.x;
    const uint32_t v = i < N ? bits[i] : 0u;
    const bool gt = i < N && v > thr, eq = i < N && v == thr;
    const unsigned m_eq = __ballot_sync(0xffffffffu, eq);
    const int2 se = warp_scan(__popc(m_eq), red);
    const bool keep = gt || (eq && se.x + __popc(m_eq & below) < eq_left);
    const unsigned m_keep = __ballot_sync(0xffffffffu, keep);
    const int2 sk = warp_scan(__popc(m_keep), red);
    if (keep) out[base + sk.x + __popc(m_keep & below)] = i;
    base += sk.y;
    eq_left -= min(eq_left, se.y);
  }
}

}  // namespace

pic_status launch_select(const SelectArgs& a, int D, int dtype, cudaStream_t st) {
  if (a.n_reqs <= 0) return PIC_OK;
  const int g_rows = (a.n_rows * a.H + 3) / 4, g_tok = (a.n_tok + 3) / 4;
#define PIC_SEL(T, DD)                                                         \
  do {                                                                        \
    if (g_rows) sel_rowstats_kernel<T, DD><<<g_rows, 128, 0, st>>>(a);        \
    if (g_tok) sel_scores_kernel<T, DD><<<g_tok, 128, 0, st>>>(a);            \
  } while (0)
  if (dtype == PIC_BF16 && D == 128) PIC_SEL(__nv_bfloat16, 128);
  else if (dtype == PIC_BF16 && D == 64) PIC_SEL(__nv_bfloat16, 64);
  else if (dtype == PIC_F32 && D == 128) PIC_SEL(float, 128);
  else if (dtype == PIC_F32 && D == 64) PIC_SEL(float, 64);
  else return fail(PIC_ERR_UNSUPPORTED, "dynamic selection: head_dim must be 64 or 128");
#undef PIC_SEL
  sel_top_kernel<<<a.n_reqs, kTopThreads, 0, st>>>(a);
  PIC_CUDA(cudaGetLastError());
  return PIC_OK;
}

}  // namespace pic
