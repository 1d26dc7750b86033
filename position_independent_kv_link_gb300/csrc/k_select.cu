// Dynamic (attention-based) choice of the prompt tokens a link recomputes: the CacheBlend-r
// step the EPIC pages measure LegoLink's static choice against (EPIC summary page: problem
// statement; Measured effects table, CacheBlend-r rows and the static-vs-dynamic row). Reading
// of the step: with the prompt linked as compiled (nothing recomputed), the query rows at layer
// 0 attend causally over the prompt and the query, RoPE at absolute positions; a prompt token's
// score is the sum of the softmax weights it receives over all query rows and heads; the
// floor(r N / 100) best-scoring tokens are recomputed (equal scores: the lower position first).
//
// Five kernels per pass, all requests at once, fp32 arithmetic, every sum in a fixed order (the
// same bits on every run):
//   sel_qrot_kernel     the query rows' q rotated to their positions and scaled by log2(e)/sqrt(D);
//   sel_logits_kernel   per block of 64 keys (prompt tokens, then the query's own keys) and KV
//                       head g: the keys rotated into shared memory, and the logits of every query
//                       row and head of g against them (query keys after a row masked);
//   sel_rowstats_kernel one warp per (query row, head): the maximum and 1 / sum of 2^(logit - max);
//   sel_scores_kernel   per block of 64 prompt tokens: each token's sum of softmax weights over
//                       heads and query rows;
//   sel_top_kernel      one CTA per request: the n-th largest score found by bisection over the
//                       scores' bit patterns, then a compaction in position order.
#include <cmath>

#include "pic_internal.h"

namespace pic {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int KB = 64;          // keys per block
constexpr int kTopThreads = 1024;

template <typename T>
__device__ __forceinline__ float kv_f(const T* p) { return to_f<T>(*p); }

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

// qrot[row][h] = RoPE(q[row][h], position n_tok + s) * log2(e) / sqrt(D); one thread per
// (row, head, rotate-half pair i).
template <int D>
__global__ void sel_qrot_kernel(SelectArgs a) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.n_rows * a.H * (D / 2)) return;
  const int i = idx % (D / 2), h = (idx / (D / 2)) % a.H, row = idx / (D / 2) / a.H;
  const SelectReq& R = a.reqs[find_req(a.n_reqs, row, [&](int k) { return a.reqs[k].row0; })];
  const float* q = a.qkv + (size_t)row * (a.H + 2 * a.G) * D + h * D;
  const float2 c = a.rope_cs[(size_t)(R.n_tok + row - R.row0) * (D / 2) + i];
  const float sc = rsqrtf((float)D) * kLog2e;
  float* o = a.qrot + ((size_t)row * a.H + h) * D;
  o[i] = (q[i] * c.x - q[i + D / 2] * c.y) * sc;
  o[i + D / 2] = (q[i + D / 2] * c.x + q[i] * c.y) * sc;
}

// CTA (key block, g): keys v = 64 kb .. of the request (v < n_tok: prompt token v from its
// page; v >= n_tok: the query's key v - n_tok from the layer-0 projections), rotated at
// position v into shared memory as [d][key]; then logits[lg0 + (s H + h)(n_tok + lq) + v] =
// qrot[s][h] . k[v] for the query rows s and the heads h of g (-inf where the key is a query
// key after row s). 256 threads: key = tid % 64, rows tid / 64 + 4 j.
template <typename T, int D>
__global__ void __launch_bounds__(256) sel_logits_kernel(SelectArgs a) {
  extern __shared__ float sm[];
  float* ks = sm;              // [D][KB]
  float* qs = sm + D * KB;     // [32][D] rows of the current chunk
  const int kb_all = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  const SelectReq& R = a.reqs[find_req(a.n_reqs, kb_all, [&](int k) { return a.reqs[k].kb0; })];
  const int nk = R.n_tok + R.lq, v0 = (kb_all - R.kb0) * KB;
  const int rep = a.H / a.G;
  // ---- the block's keys, rotated: thread = (key, quarter of the rotate-half pairs)
  {
    const int key = tid >> 2, qq = tid & 3, v = v0 + key;
    constexpr int NP = D / 8;   // pairs per quarter
    const T* src = nullptr;
    const float* srcf = nullptr;
    if (v < R.n_tok) {
      int lo = R.page0, hi = R.page0 + R.n_pages - 1;   // the token's page
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.page_pos[mid] <= v) lo = mid; else hi = mid - 1;
      }
      src = static_cast<const T*>(a.k_layer0) +
            (((size_t)a.page_block[lo] * a.G + g) * kBlock + (v - a.page_pos[lo])) * D;
    } else if (v < nk) {
      srcf = a.qkv + (size_t)(R.row0 + v - R.n_tok) * (a.H + 2 * a.G) * D + (a.H + g) * D;
    }
#pragma unroll 4
    for (int e = 0; e < NP; ++e) {
      const int i = qq * NP + e;
      float x1 = 0.f, x2 = 0.f;
      if (src) {
        x1 = kv_f<T>(src + i);
        x2 = kv_f<T>(src + i + D / 2);
      } else if (srcf) {
        x1 = srcf[i];
        x2 = srcf[i + D / 2];
      }
      float y1 = 0.f, y2 = 0.f;
      if (v < nk) {
        const float2 c = a.rope_cs[(size_t)v * (D / 2) + i];
        y1 = x1 * c.x - x2 * c.y;
        y2 = x2 * c.x + x1 * c.y;
      }
      ks[i * KB + key] = y1;
      ks[(i + D / 2) * KB + key] = y2;
    }
  }
  // ---- logits of the rows (s, h in g), 32 rows per chunk
  const int key = tid & (KB - 1), r0 = tid >> 6, v = v0 + key;
  const int n_rows = R.lq * rep;   // row j of the request: s = j / rep, h = g rep + j % rep
  for (int c0 = 0; c0 < n_rows; c0 += 32) {
    __syncthreads();   // the keys are in place; the previous chunk's rows are read
    for (int e = tid; e < 32 * D; e += 256) {
      const int j = c0 + e / D;
      const int s = j / rep, h = g * rep + j % rep;
      qs[e] = j < n_rows ? a.qrot[((size_t)(R.row0 + s) * a.H + h) * D + e % D] : 0.f;
    }
    __syncthreads();
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
#pragma unroll 8
    for (int d = 0; d < D; ++d) {
      const float kv = ks[d * KB + key];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = fmaf(qs[(r0 + 4 * u) * D + d], kv, acc[u]);
    }
    if (v < nk) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = c0 + r0 + 4 * u;
        if (j < n_rows) {
          const int s = j / rep, h = g * rep + j % rep;
          const bool masked = v >= R.n_tok && v - R.n_tok > s;
          a.logits[(size_t)R.lg0 + ((size_t)s * a.H + h) * nk + v] = masked ? -INFINITY : acc[u];
        }
      }
    }
  }
}

// One warp per (query row, head): max over its logits, and 1 / sum of 2^(logit - max).
__global__ void __launch_bounds__(128) sel_rowstats_kernel(SelectArgs a) {
  const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= a.n_rows * a.H) return;
  const int row = w / a.H, h = w % a.H;
  const SelectReq& R = a.reqs[find_req(a.n_reqs, row, [&](int k) { return a.reqs[k].row0; })];
  const int nk = R.n_tok + R.lq, s = row - R.row0;
  const float* L = a.logits + (size_t)R.lg0 + ((size_t)s * a.H + h) * nk;
  float m = -INFINITY;
  for (int v = lane; v < nk; v += 32) m = fmaxf(m, L[v]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
  for (int v = lane; v < nk; v += 32) l += exp2f(L[v] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) {
    a.ml[(size_t)w * 2] = m;
    a.ml[(size_t)w * 2 + 1] = 1.f / l;
  }
}

// CTA per block of 64 prompt tokens, 256 threads: thread (key, quarter qq) sums the weights of
// the rows j = qq, qq + 4, ... (rows in (s, h) order), then the four partial sums are added in
// quarter order.
__global__ void __launch_bounds__(256) sel_scores_kernel(SelectArgs a) {
  __shared__ float part[4][KB];
  const int kb_all = blockIdx.x, tid = threadIdx.x, key = tid & (KB - 1), qq = tid >> 6;
  const SelectReq& R = a.reqs[find_req(a.n_reqs, kb_all, [&](int k) { return a.reqs[k].pkb0; })];
  const int u = (kb_all - R.pkb0) * KB + key, nk = R.n_tok + R.lq;
  float acc = 0.f;
  if (u < R.n_tok) {
    const int n_rows = R.lq * a.H;
    for (int j = qq; j < n_rows; j += 4) {   // j = s H + h
      const size_t w = (size_t)R.row0 * a.H + j;
      acc += exp2f(a.logits[(size_t)R.lg0 + (size_t)j * nk + u] - a.ml[w * 2]) * a.ml[w * 2 + 1];
    }
  }
  part[qq][key] = acc;
  __syncthreads();
  if (qq == 0 && u < R.n_tok) a.scores[R.tok0 + u] = ((part[0][key] + part[1][key]) + part[2][key]) + part[3][key];
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

template <typename T, int D>
pic_status launch_typed(const SelectArgs& a, cudaStream_t st) {
  const int nq = a.n_rows * a.H * (D / 2);
  if (nq) sel_qrot_kernel<D><<<(nq + 255) / 256, 256, 0, st>>>(a);
  const size_t smem = (size_t)(D * KB + 32 * D) * sizeof(float);
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr[dev]) {
    PIC_CUDA(cudaFuncSetAttribute(sel_logits_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    if (dev >= 0 && dev < 64) attr[dev] = true;
  }
  if (a.n_kb) sel_logits_kernel<T, D><<<dim3(a.n_kb, a.G), 256, smem, st>>>(a);
  if (a.n_rows) sel_rowstats_kernel<<<(a.n_rows * a.H + 3) / 4, 128, 0, st>>>(a);
  if (a.n_pkb) sel_scores_kernel<<<a.n_pkb, 256, 0, st>>>(a);
  sel_top_kernel<<<a.n_reqs, kTopThreads, 0, st>>>(a);
  PIC_CUDA(cudaGetLastError());
  return PIC_OK;
}

}  // namespace

pic_status launch_select(const SelectArgs& a, int D, int dtype, cudaStream_t st) {
  if (a.n_reqs <= 0) return PIC_OK;
  if (dtype == PIC_BF16 && D == 128) return launch_typed<__nv_bfloat16, 128>(a, st);
  if (dtype == PIC_BF16 && D == 64) return launch_typed<__nv_bfloat16, 64>(a, st);
  if (dtype == PIC_F32 && D == 128) return launch_typed<float, 128>(a, st);
  if (dtype == PIC_F32 && D == 64) return launch_typed<float, 64>(a, st);
  return fail(PIC_ERR_UNSUPPORTED, "dynamic selection: head_dim must be 64 or 128");
}

}  // namespace pic
