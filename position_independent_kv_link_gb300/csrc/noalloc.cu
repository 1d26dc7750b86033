// Allocation-free variant of the kernel-level paged attention call.
//
// pic_op_attention needs device scratch (its work list and the partial results of
// page runs that are merged afterwards), and its caller supplies that buffer. Some
// callers cannot allocate device memory at all: code that runs inside a memory pool it
// does not own, plug-ins of a host program that forbids cudaMalloc after start-up, or
// paths that must not synchronize the device (cudaMalloc/cudaFree can). For them this
// file keeps a fixed scratch area in the library's own device memory and runs the same
// planner and kernels on it. The area is a file-scope device array, so every GPU that
// loads the library holds it until the process exits.
#include <cstring>
#include <mutex>
#include <vector>

#include "pic_internal.h"

using namespace pic;

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// The array's name in host code is only a host-side stand-in; the kernels need the
// device address, fetched once per device with that device current. The per-device cache is
// filled under a mutex, so first calls from several host threads are safe.
pic_status scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(PIC_ERR_UNSUPPORTED, "device index beyond the supported range");
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(PIC_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    addr[dev] = p;
  }
  *out = addr[dev];
  return PIC_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

}  // namespace

extern "C" {

size_t pic_op_attention_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

pic_status pic_op_attention_noalloc(int32_t dtype, int32_t T, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                    const void* q, const int32_t* q_pos_host, const void* k_layer,
                                    const void* v_layer, const int32_t* page_block_host,
                                    const int32_t* page_pos_host, const int32_t* page_len_host, int32_t n_pages,
                                    int32_t pool_blocks, const void* rope_cs, int32_t rope_positions, void* out,
                                    pic_stream_t stream) {
  if (T < 1 || n_pages < 1 || !q || !q_pos_host || !k_layer || !v_layer || !page_block_host || !page_pos_host ||
      !page_len_host || !rope_cs || !out || n_kv_heads < 1 || n_heads % n_kv_heads ||
      (head_dim != 64 && head_dim != 128) || (dtype != PIC_F32 && dtype != PIC_BF16) || rope_positions < 16)
    return fail(PIC_ERR_INVALID_ARG, "invalid attention arguments");
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
  in.num_sms = device_sms();
  std::vector<AttnItem> items;
  std::vector<AttnCombine> combs;
  int n_parts = 0;
  plan_attention(in, items, combs, n_parts);

  // exact footprint of this call: metadata ints, partial outputs and (max, sum) pairs, then
  // the rotated fp16 q and K of the tensor-core path
  const int rep = n_heads / n_kv_heads;
  const size_t n_ints = (size_t)T + 3 * (size_t)n_pages + kAttnItemInts * items.size() + 5 * combs.size();
  const size_t o_part = align256(n_ints * 4);
  const size_t o_ml = o_part + align256((size_t)n_parts * kAttnPartRows * rep * head_dim * 4);
  const size_t o_q16 = o_ml + align256((size_t)n_parts * kAttnPartRows * rep * 2 * 4);
  const size_t o_krot = o_q16 + (in.persistent ? align256((size_t)T * n_heads * head_dim * 2) : 0);
  const size_t o_sync = o_krot + (in.persistent ? align256(attention_krot_bytes(n_pages, n_kv_heads)) : 0);
  const size_t need = o_sync + (in.persistent ? 256 : 0);   // + the tensor-core kernel's grid-barrier counter
  if (need > kNoAllocScratchBytes)
    return fail(PIC_ERR_CAPACITY, "attention needs " + std::to_string(need) + " bytes of scratch; the fixed area holds " +
                                      std::to_string(kNoAllocScratchBytes) + " (use pic_op_attention with a caller buffer)");

  void* scratch = nullptr;
  pic_status s = scratch_address(&scratch);
  if (s != PIC_OK) return s;

  std::vector<int32_t> ints;
  ints.reserve(n_ints);
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
  // pageable source: the copy is staged before this call returns, so `ints` may go away
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
  a.part_o = (float*)((char*)scratch + o_part);
  a.part_ml = (float*)((char*)scratch + o_ml);
  a.items = (const AttnItem*)(di + o_items);
  a.n_items = (int)items.size();
  a.combines = (const AttnCombine*)(di + o_combs);
  a.n_combines = (int)combs.size();
  if (in.persistent) {
    a.n_pages = n_pages;
    s = attention_prepare_tc(a, T, pool_blocks, (__half*)((char*)scratch + o_q16), (__half*)((char*)scratch + o_krot),
                             (unsigned long long*)((char*)scratch + o_sync), st);
    if (s != PIC_OK) return s;
  }
  launch_attention(a, st);
  PIC_CUDA(cudaGetLastError());
  return PIC_OK;
}

}  // extern "C"
