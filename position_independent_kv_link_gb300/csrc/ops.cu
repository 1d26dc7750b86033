// Kernel-level C ABI: single steps of the link path (GEMM, paged attention, RoPE table)
// on caller-provided device buffers, for testing and profiling the kernels in isolation.
#include <algorithm>
#include <cstring>

#include "pic_internal.h"

using namespace pic;

namespace {

int current_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct AttnScratchLayout {
  size_t ints_bytes, part_o_off, part_ml_off, q16_off, krot_off, sync_off, total;
  int max_parts, max_items;
};

AttnScratchLayout attn_layout(int T, int n_heads, int n_kv_heads, int head_dim, int n_pages) {
  AttnScratchLayout L{};
  const int n_blocks = (T + kBlock - 1) / kBlock;
  L.max_parts = 4 * current_sms() + n_kv_heads * n_blocks;
  L.max_items = L.max_parts + n_kv_heads * n_blocks;
  const size_t ints = (size_t)T + 3 * (size_t)n_pages + kAttnItemInts * (size_t)L.max_items + 5 * (size_t)L.max_parts;
  L.ints_bytes = align256(ints * 4);
  const int rep = std::max(1, n_heads / std::max(1, n_kv_heads));
  L.part_o_off = L.ints_bytes;
  L.part_ml_off = L.part_o_off + align256((size_t)L.max_parts * kAttnPartRows * rep * head_dim * 4);
  L.q16_off = L.part_ml_off + align256((size_t)L.max_parts * kAttnPartRows * rep * 2 * 4);
  // tensor-core path: rotated fp16 q, then the rotated fp16 K of every page
  L.krot_off = L.q16_off + align256((size_t)T * n_heads * head_dim * 2);
  L.sync_off = L.krot_off + align256((size_t)n_pages * n_kv_heads * kBlock * head_dim * 2);
  L.total = L.sync_off + 256;   // the tensor-core kernel's grid-barrier counter
  return L;
}

}  // namespace

extern "C" {

pic_status pic_op_gemm(int32_t dtype, const void* W, const void* X, float* Y, int32_t N, int32_t K, int32_t T,
                       pic_stream_t stream) {
  if (!W || !X || !Y || N < 1 || K < 1 || T < 1 || (dtype != PIC_F32 && dtype != PIC_BF16))
    return fail(PIC_ERR_INVALID_ARG, "invalid gemm arguments");
  cudaStream_t st = (cudaStream_t)stream;
  PIC_CUDA(cudaMemsetAsync(Y, 0, (size_t)T * N * sizeof(float), st));
  if (dtype == PIC_BF16 && tc_gemm_supported(N, K, T)) {
    pic_status e = tc_gemm_run(W, X, Y, N, K, T, st);
    if (e != PIC_OK) return e;
  } else {
    launch_gemm_simt(dtype, false, W, X, Y, N, K, T, 1, st);
  }
  PIC_CUDA(cudaGetLastError());
  return PIC_OK;
}

pic_status pic_op_pack_weight(const void* W, void* out, int32_t N, int32_t K, pic_stream_t stream) {
  if (!W || !out || N < 1 || K < 1) return fail(PIC_ERR_INVALID_ARG, "invalid pack arguments");
  return tc_pack_weight(W, out, N, K, (cudaStream_t)stream);
}

pic_status pic_op_gemm_packed(const void* W_packed, const void* X, float* Y, int32_t N, int32_t K, int32_t T,
                              pic_stream_t stream) {
  if (!W_packed || !X || !Y || N < 1 || K < 1 || T < 1) return fail(PIC_ERR_INVALID_ARG, "invalid gemm arguments");
  if (!tc_gemm_supported(N, K, T)) return fail(PIC_ERR_UNSUPPORTED, "packed gemm: N % 128 and K % 64 must be 0");
  cudaStream_t st = (cudaStream_t)stream;
  PIC_CUDA(cudaMemsetAsync(Y, 0, (size_t)T * N * sizeof(float), st));
  return tc_gemm_run_packed(W_packed, X, Y, N, K, T, st);
}

size_t pic_op_attention_scratch_bytes(int32_t T, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                      int32_t n_pages) {
  if (T < 1 || n_heads < 1 || n_kv_heads < 1 || n_pages < 1) return 0;
  return attn_layout(T, n_heads, n_kv_heads, head_dim, n_pages).total;
}

pic_status pic_op_attention(int32_t dtype, int32_t T, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                            const void* q, const int32_t* q_pos_host, const void* k_layer, const void* v_layer,
                            const int32_t* page_block_host, const int32_t* page_pos_host,
                            const int32_t* page_len_host, int32_t n_pages, int32_t pool_blocks,
                            const void* rope_cs, int32_t rope_positions, void* out, void* scratch,
                            size_t scratch_bytes, pic_stream_t stream) {
  if (T < 1 || n_pages < 1 || !q || !q_pos_host || !k_layer || !v_layer || !page_block_host || !page_pos_host ||
      !page_len_host || !rope_cs || !out || !scratch || n_kv_heads < 1 || n_heads % n_kv_heads ||
      (head_dim != 64 && head_dim != 128) || (dtype != PIC_F32 && dtype != PIC_BF16) || rope_positions < 16)
    return fail(PIC_ERR_INVALID_ARG, "invalid attention arguments");
  const AttnScratchLayout L = attn_layout(T, n_heads, n_kv_heads, head_dim, n_pages);
  if (scratch_bytes < L.total) return fail(PIC_ERR_INVALID_ARG, "attention scratch too small");
  for (int t = 0; t < T; ++t)
    if (q_pos_host[t] < 0 || q_pos_host[t] >= rope_positions || (t && q_pos_host[t] <= q_pos_host[t - 1]))
      return fail(PIC_ERR_INVALID_ARG, "query positions must be ascending and inside the RoPE table");
  for (int p = 0; p < n_pages; ++p)
    if (page_block_host[p] < 0 || page_block_host[p] >= pool_blocks || page_len_host[p] < 1 ||
        page_len_host[p] > kBlock || page_pos_host[p] < 0 ||
        page_pos_host[p] + page_len_host[p] > rope_positions ||
        (p && page_pos_host[p] < page_pos_host[p - 1] + page_len_host[p - 1]))
      return fail(PIC_ERR_INVALID_ARG,
                  "pages must be in position order, inside the pool and RoPE table, with 1..16 valid rows");
  std::vector<int> row_pos(q_pos_host, q_pos_host + T), ppos(page_pos_host, page_pos_host + n_pages);
  AttnPlanInput in;
  in.seq_row_begin = {0};
  in.seq_row_end = {T};
  in.seq_page_begin = {0};
  in.seq_page_end = {n_pages};
  in.row_pos = &row_pos;
  in.page_pos = &ppos;
  in.G = n_kv_heads;
  in.rows_per_block = attention_rows_per_block(dtype, head_dim, n_heads / n_kv_heads);
  in.persistent = attention_persistent(dtype, head_dim, n_heads / n_kv_heads);
  in.num_sms = current_sms();
  std::vector<AttnItem> items;
  std::vector<AttnCombine> combs;
  int n_parts = 0;
  plan_attention(in, items, combs, n_parts);
  if (n_parts > L.max_parts || (int)items.size() > L.max_items)
    return fail(PIC_ERR_CAPACITY, "attention plan exceeds its scratch bound");
  std::vector<int32_t> ints;
  ints.insert(ints.end(), q_pos_host, q_pos_host + T);
  ints.insert(ints.end(), page_block_host, page_block_host + n_pages);
  ints.insert(ints.end(), page_pos_host, page_pos_host + n_pages);
  ints.insert(ints.end(), page_len_host, page_len_host + n_pages);
  const size_t o_items = ints.size();
  ints.resize(o_items + items.size() * kAttnItemInts);
  std::memcpy(ints.data() + o_items, items.data(), items.size() * sizeof(AttnItem));
  const size_t o_combs = ints.size();
  ints.resize(o_combs + combs.size() * 5);
  std::memcpy(ints.data() + o_combs, combs.data(), combs.size() * sizeof(AttnCombine));
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* di = (int32_t*)scratch;
  PIC_CUDA(cudaMemcpyAsync(di, ints.data(), ints.size() * 4, cudaMemcpyHostToDevice, st));
  AttnArgs a{};
  a.dtype = dtype;
  a.rb = in.rows_per_block;
  a.H = n_heads;
  a.G = n_kv_heads;
  a.D = head_dim;
  a.q = (const float*)q;
  a.q_pos = di;
  a.k_layer = k_layer;
  a.v_layer = v_layer;
  a.page_block = di + T;
  a.page_pos = di + T + n_pages;
  a.page_len = di + T + 2 * n_pages;
  a.rope_cs = (const float2*)rope_cs;
  a.out = out;
  a.part_o = (float*)((char*)scratch + L.part_o_off);
  a.part_ml = (float*)((char*)scratch + L.part_ml_off);
  a.items = (const AttnItem*)(di + o_items);
  a.n_items = (int)items.size();
  a.combines = (const AttnCombine*)(di + o_combs);
  a.n_combines = (int)combs.size();
  if (in.persistent) {
    a.n_pages = n_pages;
    pic_status e = attention_prepare_tc(a, T, pool_blocks, (__half*)((char*)scratch + L.q16_off),
                                        (__half*)((char*)scratch + L.krot_off),
                                        (unsigned long long*)((char*)scratch + L.sync_off), st);
    if (e != PIC_OK) return e;
  }
  launch_attention(a, st);
  PIC_CUDA(cudaGetLastError());
  return PIC_OK;
}

pic_status pic_op_attention_plan(int32_t dtype, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                 int32_t n_seqs, const int32_t* seq_rows, const int32_t* seq_pages,
                                 const int32_t* row_pos, const int32_t* page_pos, int32_t num_sms, int32_t* items,
                                 int32_t max_items, int32_t* combines, int32_t max_combines, int32_t* counts) {
  if (n_seqs < 1 || !seq_rows || !seq_pages || !counts || num_sms < 1 || n_kv_heads < 1 || n_heads < 1 ||
      n_heads % n_kv_heads || (head_dim != 64 && head_dim != 128) || (dtype != PIC_F32 && dtype != PIC_BF16) ||
      max_items < 0 || max_combines < 0 || (max_items > 0 && !items) || (max_combines > 0 && !combines) ||
      seq_rows[0] != 0 || seq_pages[0] != 0)
    return fail(PIC_ERR_INVALID_ARG, "invalid plan arguments");
  for (int s = 0; s < n_seqs; ++s) {
    if (seq_rows[s + 1] < seq_rows[s] || seq_pages[s + 1] < seq_pages[s])
      return fail(PIC_ERR_INVALID_ARG, "sequence offsets must not decrease");
    for (int r = seq_rows[s] + 1; r < seq_rows[s + 1]; ++r)
      if (row_pos[r] <= row_pos[r - 1]) return fail(PIC_ERR_INVALID_ARG, "row positions must ascend per sequence");
    for (int p = seq_pages[s] + 1; p < seq_pages[s + 1]; ++p)
      if (page_pos[p] <= page_pos[p - 1]) return fail(PIC_ERR_INVALID_ARG, "page positions must ascend per sequence");
  }
  if ((seq_rows[n_seqs] > 0 && !row_pos) || (seq_pages[n_seqs] > 0 && !page_pos))
    return fail(PIC_ERR_INVALID_ARG, "invalid plan arguments");
  std::vector<int> rp(row_pos, row_pos + seq_rows[n_seqs]), pp(page_pos, page_pos + seq_pages[n_seqs]);
  AttnPlanInput in;
  for (int s = 0; s < n_seqs; ++s) {
    in.seq_row_begin.push_back(seq_rows[s]);
    in.seq_row_end.push_back(seq_rows[s + 1]);
    in.seq_page_begin.push_back(seq_pages[s]);
    in.seq_page_end.push_back(seq_pages[s + 1]);
  }
  in.row_pos = &rp;
  in.page_pos = &pp;
  in.G = n_kv_heads;
  in.num_sms = num_sms;
  in.rows_per_block = attention_rows_per_block(dtype, head_dim, n_heads / n_kv_heads);
  in.persistent = attention_persistent(dtype, head_dim, n_heads / n_kv_heads);
  std::vector<AttnItem> its;
  std::vector<AttnCombine> cbs;
  int n_parts = 0;
  plan_attention(in, its, cbs, n_parts);
  counts[0] = (int32_t)its.size();
  counts[1] = (int32_t)cbs.size();
  counts[2] = n_parts;
  if ((int)its.size() > max_items || (int)cbs.size() > max_combines)
    return fail(PIC_ERR_CAPACITY, "plan output arrays too small");
  if (!its.empty()) std::memcpy(items, its.data(), its.size() * sizeof(AttnItem));
  if (!cbs.empty()) std::memcpy(combines, cbs.data(), cbs.size() * sizeof(AttnCombine));
  return PIC_OK;
}

pic_status pic_op_rope_table(int32_t n_pos, int32_t head_dim, double base, void* out, pic_stream_t stream) {
  if (n_pos < 1 || head_dim < 2 || head_dim % 2 || !out || !(base > 1.0))
    return fail(PIC_ERR_INVALID_ARG, "invalid rope table arguments");
  std::vector<float2> tab;
  rope_table_host(n_pos, head_dim, base, tab);
  PIC_CUDA(cudaMemcpyAsync(out, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice,
                           (cudaStream_t)stream));
  PIC_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  return PIC_OK;
}

}  // extern "C"
