// Sparse-query paged attention with RoPE fused at load (MEPIC abstract: K is kept
// without positional encoding and rotated inside the attention kernel), causal by
// absolute position, GQA head sharing, split over page ranges with an LSE merge.
//
// This file holds the generic warp-per-(row, head) kernel (any dtype, D = 64 or 128),
// the split merge and the host planner. The bf16 D=128 kernels take the same work
// items: k_attn_tc.cu (tcgen05, 4 query heads per KV head) and k_attn_mma.cu
// (mma.sync, 1, 2 or 8 query heads per KV head).
#include <algorithm>
#include <cmath>

#include "pic_internal.h"

namespace pic {

void launch_attention_mma(const AttnArgs& a, cudaStream_t st);  // k_attn_mma.cu
bool tc_attention_supported(int dtype, int D, int rep);          // k_attn_tc.cu
void launch_attention_tc(const AttnArgs& a, cudaStream_t st);

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// T: KV storage type; O: output type (fp16 for bf16 KV, fp32 for fp32 KV); q is fp32.
template <typename T, typename O, int D>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnArgs a) {
  constexpr int NJ = D / 32;   // dims per lane: lane + 32 j
  const AttnItem it = a.items[blockIdx.x];
  const int rep = a.H / a.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* Q = a.q;
  const T* Kl = (const T*)a.k_layer;
  const T* Vl = (const T*)a.v_layer;
  const float scale = rsqrtf((float)D) * kLog2e;
  for (int pr = warp; pr < it.nrows * rep; pr += 4) {
    const int r = pr / rep, hh = pr % rep;
    const int t = it.row0 + r, h = it.g * rep + hh;
    const int qp = a.q_pos[t];
    float q[NJ], o[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      q[j] = Q[((size_t)t * a.H + h) * D + lane + 32 * j];
      o[j] = 0.f;
    }
    const float2* csq = a.rope_cs + (size_t)qp * (D / 2);
#pragma unroll
    for (int j = 0; j < NJ / 2; ++j) {
      const float2 cs = csq[lane + 32 * j];
      const float x1 = q[j], x2 = q[j + NJ / 2];
      q[j] = (x1 * cs.x - x2 * cs.y) * scale;
      q[j + NJ / 2] = (x2 * cs.x + x1 * cs.y) * scale;
    }
    float m = -INFINITY, l = 0.f;
    bool done = false;
    for (int p = it.page0; p < it.page1 && !done; ++p) {
      const int blk = a.page_block[p], base = a.page_pos[p], len = a.page_len[p];
      for (int rr = 0; rr < len; ++rr) {
        const int kp = base + rr;
        if (kp > qp) { done = true; break; }
        const size_t off = (((size_t)blk * a.G + it.g) * kBlock + rr) * D;
        const float2* csk = a.rope_cs + (size_t)kp * (D / 2);
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < NJ / 2; ++j) {
          const float2 cs = csk[lane + 32 * j];
          const float k1 = to_f<T>(Kl[off + lane + 32 * j]);
          const float k2 = to_f<T>(Kl[off + lane + 32 * (j + NJ / 2)]);
          s += q[j] * (k1 * cs.x - k2 * cs.y) + q[j + NJ / 2] * (k2 * cs.x + k1 * cs.y);
        }
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) s += __shfl_xor_sync(0xffffffffu, s, x);
        const float mn = fmaxf(m, s);
        const float corr = exp2f(m - mn);
        const float pw = exp2f(s - mn);
        l = l * corr + pw;
#pragma unroll
        for (int j = 0; j < NJ; ++j) o[j] = o[j] * corr + pw * to_f<T>(Vl[off + lane + 32 * j]);
        m = mn;
      }
    }
    if (it.part < 0) {
      const float inv = 1.f / l;
      O* out = (O*)a.out;
#pragma unroll
      for (int j = 0; j < NJ; ++j) out[((size_t)t * a.H + h) * D + lane + 32 * j] = from_f<O>(o[j] * inv);
    } else {
      const size_t pi = ((size_t)it.part * kAttnPartRows + r) * rep + hh;
#pragma unroll
      for (int j = 0; j < NJ; ++j) a.part_o[pi * D + lane + 32 * j] = o[j];
      if (lane == 0) {
        a.part_ml[pi * 2] = m;
        a.part_ml[pi * 2 + 1] = l;
      }
    }
  }
}

// Merge split results: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s with M = max_s m_s
// over the parts that saw a key (l_s > 0). grid (merges, ceil(rows * rep / 8)); one warp per
// (row, head). The lanes first read the parts' (m, l) side by side (32 parts per pass) and
// reduce M and the denominator across the warp; then each lane sums its D/32 dims over the
// parts with the weights broadcast, the parts' loads independent of each other.
template <typename O, int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a) {
  pdl_enter();
  constexpr int NJ = D / 32;
  const AttnCombine c = a.combines[blockIdx.x];
  const int rep = a.H / a.G;
  const int pr = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (pr >= c.nrows * rep) return;
  const int r = pr / rep, hh = pr % rep;
  auto part = [&](int s) { return ((size_t)(c.part0 + s) * kAttnPartRows + r) * rep + hh; };
  float M = -INFINITY;
  for (int s0 = 0; s0 < c.nparts; s0 += 32) {
    const int s = s0 + lane;
    if (s < c.nparts) {
      const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + part(s) * 2);
      if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float o[NJ], L = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) o[j] = 0.f;
  for (int s0 = 0; s0 < c.nparts; s0 += 32) {
    const int s = s0 + lane;
    float w = 0.f;   // this lane's part weight
    if (s < c.nparts) {
      const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + part(s) * 2);
      if (ml.y > 0.f) {
        // fp32 partials hold the part's unnormalized sum (reference max ml.x); fp16 partials
        // hold it divided by the part's own sum ml.y
        w = a.part_f16 ? exp2f(ml.x - M) * ml.y : exp2f(ml.x - M);
        L += a.part_f16 ? w : w * ml.y;
      }
    }
    const int n = min(32, c.nparts - s0);
    if (a.part_f16) {
#pragma unroll 4
      for (int k = 0; k < n; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        const __half* src = reinterpret_cast<const __half*>(a.part_o) + part(s0 + k) * D + lane * NJ;
        if constexpr (NJ == 4) {
          const uint2 u = *reinterpret_cast<const uint2*>(src);
          const float2 x0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
          const float2 x1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
          o[0] += wk * x0.x, o[1] += wk * x0.y, o[2] += wk * x1.x, o[3] += wk * x1.y;
        } else {
          const float2 x = __half22float2(*reinterpret_cast<const __half2*>(src));
          o[0] += wk * x.x, o[1] += wk * x.y;
        }
      }
    } else {
#pragma unroll 4
      for (int k = 0; k < n; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        const float* src = a.part_o + part(s0 + k) * D + lane * NJ;
        if constexpr (NJ == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          o[0] += wk * x.x, o[1] += wk * x.y, o[2] += wk * x.z, o[3] += wk * x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src);
          o[0] += wk * x.x, o[1] += wk * x.y;
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const int t = c.row0 + r, h = c.g * rep + hh;
  const float inv = L > 0.f ? 1.f / L : 0.f;
  O* out = (O*)a.out + ((size_t)t * a.H + h) * D + lane * NJ;
#pragma unroll
  for (int j = 0; j < NJ; ++j) out[j] = from_f<O>(o[j] * inv);
}

template <typename T, typename O, int D>
void launch_simt(const AttnArgs& a, cudaStream_t st) {
  if (a.n_items > 0) attn_simt_kernel<T, O, D><<<a.n_items, 128, 0, st>>>(a);
  if (a.n_combines > 0) {
    const int rep = a.H / a.G;
    launch_dependent(attn_combine_kernel<O, D>, dim3(a.n_combines, (a.rb * rep + 7) / 8), dim3(256), 0, st, a);
  }
}

}  // namespace

void launch_attention_simt(const AttnArgs& a, cudaStream_t st) {
  if (a.dtype == PIC_BF16) {
    if (a.D == 128) launch_simt<__nv_bfloat16, __half, 128>(a, st);
    else launch_simt<__nv_bfloat16, __half, 64>(a, st);
  } else {
    if (a.D == 128) launch_simt<float, float, 128>(a, st);
    else launch_simt<float, float, 64>(a, st);
  }
}

bool use_mma(int dtype, int D, int rep) { return dtype == PIC_BF16 && D == 128 && (rep == 1 || rep == 2 || rep == 4 || rep == 8); }

int attention_rows_per_block(int dtype, int D, int rep) {
  if (tc_attention_supported(dtype, D, rep)) return attention_tc_rows_per_item();
  return (use_mma(dtype, D, rep) && rep <= 4) ? 32 : 16;
}

bool attention_persistent(int dtype, int D, int rep) { return tc_attention_supported(dtype, D, rep); }

pic_status attention_prepare_tc(AttnArgs& a, int T, int pool_blocks, __half* q16, __half* krot,
                                unsigned long long* sync, cudaStream_t st) {
  launch_rope_q16(T, a.H, a.q, a.q_pos, a.rope_cs, q16, st);
  PIC_CUDA(cudaMemsetAsync(sync, 0, sizeof(*sync), st));
  a.q16 = q16;
  a.krot = krot;
  a.grid_sync = sync;
  a.sync_base = 0;
  if (!attn_v_map(&a.vmap, &a.vmap1, a.v_layer, pool_blocks, a.G) || !attn_krot_map(&a.kmap, krot, a.n_pages, a.G))
    return fail(PIC_ERR_CUDA, "cuTensorMapEncodeTiled failed for the attention operands");
  return PIC_OK;
}

void launch_attention(const AttnArgs& a, cudaStream_t st) {
  if (tc_attention_supported(a.dtype, a.D, a.H / a.G)) {
    AttnArgs b = a;
    b.part_f16 = 1;
    launch_attention_tc(b, st);
    if (b.n_combines > 0) {
      b.n_items = 0;  // merge only
      launch_attention_simt(b, st);
    }
  } else if (use_mma(a.dtype, a.D, a.H / a.G))
    launch_attention_mma(a, st);
  else
    launch_attention_simt(a, st);
}

size_t attention_part_bytes(int n_parts, int rep, int D) {
  return (size_t)n_parts * kAttnPartRows * rep * (D + 2) * sizeof(float);
}

// Blocks of <= rows_per_block consecutive rows of one sequence; each block reads the prefix of the
// sequence's pages up to its last row's position, cut into runs of P pages (P chosen below).
// For blocks of more than 32 rows, the pages its first 32 rows see end earlier (pe0): every
// item records where, clipped to its own run (page_mid).
void plan_attention(const AttnPlanInput& in, std::vector<AttnItem>& items, std::vector<AttnCombine>& combines,
                    int& n_parts) {
  struct Blk { int row0, nrows, pb, pe, pe0; };
  std::vector<Blk> blks;
  long long total = 0;
  const std::vector<int>& rp = *in.row_pos;
  const std::vector<int>& pp = *in.page_pos;
  for (size_t s = 0; s < in.seq_row_begin.size(); ++s) {
    const int rb = in.rows_per_block > 0 ? in.rows_per_block : kBlock;
    for (int r0 = in.seq_row_begin[s]; r0 < in.seq_row_end[s]; r0 += rb) {
      const int n = std::min(rb, in.seq_row_end[s] - r0);
      auto visible_end = [&](int last_row) {
        int pe = in.seq_page_begin[s];
        while (pe < in.seq_page_end[s] && pp[pe] <= rp[last_row]) ++pe;
        return pe;
      };
      const int pe = visible_end(r0 + n - 1);
      const int pe0 = n > 32 ? visible_end(r0 + 31) : pe;
      blks.push_back({r0, n, in.seq_page_begin[s], pe, pe0});
      total += (long long)(pe - in.seq_page_begin[s]);
    }
  }
  const int G = std::max(1, in.G);
  auto build = [&](int P, std::vector<AttnItem>& its, std::vector<AttnCombine>& cbs, int& nparts) {
    its.clear();
    cbs.clear();
    nparts = 0;
    for (const Blk& b : blks) {
      const int np = b.pe - b.pb;
      const int ns = std::max(1, (np + P - 1) / P);
      for (int g = 0; g < in.G; ++g) {
        if (ns == 1) {
          its.push_back({b.row0, b.nrows, g, b.pb, b.pe, -1, b.pe0});
          continue;
        }
        cbs.push_back({b.row0, b.nrows, g, nparts, ns});
        for (int s = 0; s < ns; ++s) {
          const int p0 = b.pb + s * P, p1 = std::min(b.pe, p0 + P);
          its.push_back({b.row0, b.nrows, g, p0, p1, nparts + s, std::min(p1, std::max(p0, b.pe0))});
        }
        nparts += ns;
      }
    }
    // Heaviest items first so the long ranges start early.
    std::stable_sort(its.begin(), its.end(),
                     [](const AttnItem& x, const AttnItem& y) { return (x.page1 - x.page0) > (y.page1 - y.page0); });
  };
  if (!in.persistent) {
    // Pages per split part: one CTA per item, about four items per SM, never finer than 4 pages.
    const long long target = std::max<long long>(1, 4LL * in.num_sms / G);
    build((int)std::max<long long>(4, (total + target - 1) / target), items, combines, n_parts);
    return;
  }
  // Persistent kernel: CTA c of n = min(items, SMs) takes items c, c + n, c + 2n, ...; the sorted
  // items are dealt in snake order (round k runs over the CTAs backwards when k is odd). Parts are
  // whole 64-key tiles (4 pages). Candidate part sizes, for about 1, 1.5, 2, 3 and 4 items per
  // SM: the size from the average page count, and the smallest size whose item count does not
  // exceed the target (blocks seldom divide evenly: at the 8B 10 x 512 link the first gives 168
  // items for 152 SMs, the second exactly 152). The candidate with the smallest estimate is
  // taken (then the fewest items, then the smaller size). The estimate is the deal's makespan
  // times the SM count plus kMergeCost per split part: each part's fp16 partial is written by its
  // item and read back by the merge kernel, which runs over all SMs. An item's cost, in units of
  // 0.01 us, is a fit of this kernel's per-CTA globaltimer traces on GB300: 26 per 64-key tile,
  // 33 per MMA tile that takes part in it (rows 0-31 up to page_mid, rows 32-63 throughout), and
  // 491 per item (Q load, pipeline fill, O drain).
  constexpr long long kMergeCost = 150;
  auto cost = [](const AttnItem& it) -> long long {
    const int nt = (it.page1 - it.page0 + 3) / 4;
    const int n0 = std::max(0, (it.page_mid - it.page0 + 3) / 4), n1 = it.nrows > 32 ? nt : 0;
    return 26LL * nt + 33LL * (n0 + n1) + 491;
  };
  auto deal = [&](std::vector<AttnItem>& its) -> long long {
    const int n = std::min<int>((int)its.size(), std::max(1, in.num_sms));
    std::vector<AttnItem> dealt(its.size());
    std::vector<long long> load(std::max(1, n), 0);
    for (size_t k = 0; k * n < its.size(); ++k) {
      const int m = (int)std::min<size_t>(n, its.size() - k * n);
      for (int c = 0; c < m; ++c) {
        const AttnItem& it = its[k * n + ((k & 1) ? m - 1 - c : c)];
        dealt[k * n + c] = it;
        load[c] += cost(it);
      }
    }
    its.swap(dealt);
    return *std::max_element(load.begin(), load.end());
  };
  int max_pages = 1;
  for (const Blk& b : blks) max_pages = std::max(max_pages, b.pe - b.pb);
  auto n_items_of = [&](int P) {
    long long n = 0;
    for (const Blk& b : blks) n += std::max(1, (b.pe - b.pb + P - 1) / P);
    return n * G;
  };
  std::vector<int> cands;
  for (const int twice_per_sm : {2, 3, 4, 6, 8}) {
    const long long want = std::max<long long>(1, (long long)twice_per_sm * std::max(1, in.num_sms) / 2);
    int P = (int)((std::max<long long>(8, (total * G + want - 1) / want) + 3) / 4 * 4);
    cands.push_back(P);
    while (n_items_of(P) > want && P < max_pages) P += 4;
    cands.push_back(P);
  }
  std::sort(cands.begin(), cands.end());
  cands.erase(std::unique(cands.begin(), cands.end()), cands.end());
  long long best = -1;
  for (const int P : cands) {
    std::vector<AttnItem> its;
    std::vector<AttnCombine> cbs;
    int nparts = 0;
    build(P, its, cbs, nparts);
    const long long est = deal(its) * std::max(1, in.num_sms) + kMergeCost * nparts;
    if (best < 0 || est < best || (est == best && its.size() < items.size())) {
      best = est;
      items.swap(its);
      combines.swap(cbs);
      n_parts = nparts;
    }
  }
}

void rope_table_host(int n_pos, int D, double base, std::vector<float2>& out) {
  const int h = D / 2;
  out.resize((size_t)n_pos * h);
  std::vector<double> theta(h);
  for (int i = 0; i < h; ++i) theta[i] = std::pow(base, -2.0 * i / D);
  for (int p = 0; p < n_pos; ++p)
    for (int i = 0; i < h; ++i) {
      const double ang = (double)p * theta[i];
      out[(size_t)p * h + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
}

}  // namespace pic
