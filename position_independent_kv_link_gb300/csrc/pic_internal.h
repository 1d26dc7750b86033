// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "pic.h"

namespace pic {

constexpr int kBlock = 16;  // tokens per KV page

// ------------------------------------------------------------------ error plumbing
void set_error(const std::string& msg);
pic_status fail(pic_status s, const std::string& msg);
#define PIC_CUDA(call)                                                                \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess)                                                            \
      return ::pic::fail(PIC_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

// ------------------------------------------------------------------ programmatic dependent launch
// The forward's kernels are launched as programmatic dependents of the kernel before them in
// the stream, so a kernel's launch and prologue overlap the previous kernel's tail. Such a
// kernel calls pdl_enter() before its first global-memory access: it waits until the
// previous kernel has completed and its writes are visible, then lets the next kernel launch.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
}
template <typename... P, typename... A>
inline cudaError_t launch_dependent(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    A... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<P>(args)...);
}

// ------------------------------------------------------------------ element helpers
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }

// Storage of weights and KV follows the model dtype. For bf16 models the activations fed
// to the tensor cores (normed hidden rows, attention output, SwiGLU output) are fp16 and
// the packed weight copy is fp16 too (every bf16 weight above 2^-14 in magnitude is exact
// in fp16): 3 more mantissa bits per rounding at the same tensor-core rate. Accumulators,
// norms, softmax and the residual stream are fp32 throughout; q stays fp32 until RoPE.
inline size_t dtype_size(int dtype) { return dtype == PIC_BF16 ? 2 : 4; }
inline size_t act_size(int dtype) { return dtype == PIC_BF16 ? 2 : 4; }

// ------------------------------------------------------------------ row-wise kernels (k_rows.cu)
// h[t] = E[tok[t]] (fp32); x[t] = RMSNorm(h[t]) * gain in the activation type.
void launch_embed_norm(int dtype, int T, int d, const void* embed, const int* tok, const float* gain, float eps,
                       float* h, void* x, cudaStream_t st);
// QKV epilogue: reads the fp32 accumulator [T][(H+2G)D], writes the pre-RoPE
// k, v rows (model dtype) into their page slots of one layer, and q [T][H][D]: fp32 pre-RoPE
// when q16 is null, else (q16 non-null, D = 128) rotated at pos[t] with the cos/sin table,
// times log2(e)/sqrt(D), in fp16 into q16 -- the operand of the tensor-core attention.
void launch_qkv_epilogue(int dtype, int T, int H, int G, int D, float* acc, float* q, const int* slot, void* k_layer,
                         void* v_layer, const int* pos, const float2* rope_cs, __half* q16, cudaStream_t st);
// q16[t][h] = fp16(RoPE(q[t][h], pos[t]) * log2(e)/sqrt(D)) for D = 128 (same arithmetic as the
// epilogue's q16 output), for callers that hold fp32 pre-RoPE q.
void launch_rope_q16(int T, int H, const float* q, const int* pos, const float2* rope_cs, __half* q16,
                     cudaStream_t st);
// y = RMSNorm(h[t]) * gain. Not final: x[t] = y (activation type). Final: hidden_out[out_row[t]]
// = y (fp32) when out_row[t] >= 0 and lm_x[lg_row[t]] = y (activation type) when lg_row[t] >= 0.
void launch_rmsnorm_rows(int dtype, int T, int d, const float* h, const float* gain, float eps, void* x,
                         bool final_layer, const int* out_row, float* hidden_out, const int* lg_row, void* lm_x,
                         cudaStream_t st);
// act[t][j] = silu(gate) * up (activation type) from the accumulator [T][2F] (gate cols, then
// up cols).
void launch_swiglu(int dtype, int T, int F, float* acc, void* act, cudaStream_t st);
// n floats at p (and n2 at p2, when given) set to zero, in one launch (a forward kernel:
// programmatic dependent launch).
void launch_zero(float* p, size_t n, cudaStream_t st, float* p2 = nullptr, size_t n2 = 0);
// For each pair i: copy block src[i] -> dst[i] in every layer of both pools.
void launch_copy_blocks(int n_pairs, const int* pairs, int n_layers, int num_blocks_total, size_t block_bytes,
                        void* k_pool, void* v_pool, cudaStream_t st);
// Copies rows [n_layers][n][G][D] of a chunk's KV into its pages (row t -> blocks[t/16], t%16).
void launch_import_kv(int dtype, int n_layers, int n, int G, int D, const void* k_src, const void* v_src,
                      const int* blocks, int num_blocks_total, void* k_pool, void* v_pool, cudaStream_t st);

// ------------------------------------------------------------------ GEMMs
// Y[T][N] (fp32) += X[T][K] . W[N][K]^T; K split evenly over `splits` CTAs (atomic adds).
// W in `w_dtype` (PIC_F32 / PIC_BF16); X in `x_half` ? fp16 : the same type as W.
void launch_gemm_simt(int w_dtype, bool x_half, const void* W, const void* X, float* Y, int N, int K, int T,
                      int splits, cudaStream_t st);

// Shape rules of the tcgen05 kernel (N % 128 == 0, K % 64 == 0).
bool tc_gemm_supported(int N, int K, int T);
// Y[T][N] (fp32, 16-byte aligned) += X[T][K] . W[N][K]^T on tcgen05 (persistent stream-K),
// W and X bf16.
pic_status tc_gemm_run(const void* W, const void* X, float* Y, int N, int K, int T, cudaStream_t st);
// Scale folded into the fp16 q operand of the tensor-core attention: log2(e) / sqrt(128).
constexpr float kQ16Scale = 1.4426950408889634f * 0.08838834764831845f;

// Same with fp16 weights in the tile layout written by tc_pack_weight and fp16 X.
// early_weights: launch as a programmatic dependent of the previous kernel, streaming weight
// tiles before that kernel completes -- only for weights no kernel in flight writes.
// tile_ready (non-null): Y = X . W^T instead of Y += ...: the kernel zeroes Y's tiles itself,
// publishing each in tile_ready[tile] (>= tc_gemm_tiles(N, T) ints, device) as `epoch`, which
// must differ from the value any earlier launch left there.
pic_status tc_gemm_run_packed(const void* Wp, const void* X, float* Y, int N, int K, int T, cudaStream_t st,
                              bool early_weights = false, int* tile_ready = nullptr, uint32_t epoch = 0);
size_t tc_gemm_tiles(int N, int T);
// [N][K] bf16 -> N*K*2 bytes of fp16 16 KB tiles (128 rows x 64 k, 128-byte swizzled image),
// tile (mt, kb) at (mt * K/64 + kb) * 16 KB.
pic_status tc_pack_weight(const void* W, void* out, int N, int K, cudaStream_t st);
// Reads and clears the device flag set when a tcgen05 GEMM gave up a bounded wait.
pic_status tc_check_timeout();
// Same for the tcgen05 attention kernel (k_attn_tc.cu).
pic_status attn_check_timeout();
// Reads and clears the device word the row-wise kernels set when a value bound for an fp16
// tensor-core operand is outside fp16's range (k_rows.cu): PIC_ERR_RANGE.
pic_status rows_check_range();
// Reads and clears the flag tc_pack_weight sets for a weight outside fp16's range: PIC_ERR_RANGE.
pic_status tc_check_pack_range();
// Set those device flags from the host, as the kernels would (pic_debug_raise_device_flag).
void attn_raise_timeout();
void tc_raise_timeout();
void rows_raise_range();

// ------------------------------------------------------------------ attention (k_attn.cu)
constexpr int kAttnPartRows = 64;          // row slots of one split-partial slab (rows of the largest item)

// One CTA's work: <= rb consecutive rows of one sequence x one KV head x the page range
// [page0, page1). part < 0: write the normalized output directly, else a split partial.
// page_mid: the first 32 rows of the item see no key at or after page page_mid of the range
// (the tensor-core kernel stops their MMA tile there); page1 when the item has <= 32 rows.
struct AttnItem {
  int row0, nrows, g, page0, page1, part, page_mid;
};
constexpr int kAttnItemInts = sizeof(AttnItem) / sizeof(int);
struct AttnCombine {   // merge `nparts` partial results of rows [row0, row0+nrows) for KV head g
  int row0, nrows, g, part0, nparts;
};
struct AttnArgs {
  // tensor-core kernel only (attention_persistent shapes): the kernel first rotates the K of the
  // n_pages pages into the scratch krot [n_pages][G][16][128] fp16, which kmap boxes 4
  // consecutive pages of (attn_krot_map); vmap / vmap1 box one 64-dim half of 4 consecutive
  // blocks' / one block's page of the V pool layer (attn_v_map); q16: q as fp16 [T][H][D],
  // rotated and scaled (the QKV epilogue's q16 output). grid_sync: a device counter the CTAs
  // add 1 to at the kernel's grid barrier, which opens once it reaches sync_base + the grid size
  // (the caller adds attention_tc_grid(n_items) to sync_base after each launch).
  CUtensorMap kmap, vmap, vmap1;
  __half* krot;
  int n_pages;
  unsigned long long* grid_sync;
  unsigned long long sync_base;
  const __half* q16;
  int dtype, H, G, D;
  int rb;                   // rows per work item of this plan (16, 32 or 64)
  const float* q;           // [T][H][D] pre-RoPE, fp32
  const int* q_pos;         // [T]
  const void* k_layer;      // [nb][G][16][D]
  const void* v_layer;
  const int* page_block;    // flattened pages of all sequences
  const int* page_pos;
  const int* page_len;
  const float2* rope_cs;    // [max_pos][D/2]
  void* out;                // [T][H][D] activation type (fp16 for bf16 KV, fp32 for fp32 KV)
  float* part_o;            // [parts][kAttnPartRows][rep][D]: fp32 unnormalized sums, or (part_f16) fp16 O / l
  int part_f16;             // the tensor-core kernel writes its split partials normalized, in fp16
  float* part_ml;           // [parts][kAttnPartRows][rep][2]
  const AttnItem* items;
  int n_items;
  const AttnCombine* combines;
  int n_combines;
};
void launch_attention(const AttnArgs& a, cudaStream_t st);

// Host-side planning shared by link/compile and the kernel-level call.
struct AttnPlanInput {
  // per sequence: [row_begin, row_end) rows (ascending positions) and [page_begin, page_end)
  std::vector<int> seq_row_begin, seq_row_end, seq_page_begin, seq_page_end;
  const std::vector<int>* row_pos;
  const std::vector<int>* page_pos;
  int G;
  int num_sms;
  int rows_per_block;       // from attention_rows_per_block()
  bool persistent = false;  // from attention_persistent(): one CTA per SM walks a strided item list
};
// Rows per work item the attention kernels take for this model shape (16, 32, or 64 for the
// tensor-core kernel, whose items are two MMA tiles of 32 rows).
int attention_rows_per_block(int dtype, int D, int rep);
int attention_tc_rows_per_item();   // k_attn_tc.cu
// True when the shape runs the persistent tensor-core kernel: its CTA b takes items b, b + grid,
// b + 2 grid, ... with grid = min(items, SMs), so the planner orders items for that walk.
bool attention_persistent(int dtype, int D, int rep);
// Tensor maps of the tensor-core attention (k_attn_tc.cu): the V pool layer [pool_blocks][G][16]
// [128] bf16 viewed as 5-D (64 dims, 2 halves, 16 rows, G, blocks) -- m4 boxes one half of the
// pages of 4 consecutive blocks of one KV head (8 KB), m1 one half of one page (2 KB) -- and the
// rotated-K scratch [n_pages][G][16][128] fp16 the same way with 4-page boxes. 128-byte
// swizzled. False when encoding fails.
bool attn_v_map(CUtensorMap* m4, CUtensorMap* m1, const void* v_layer, int pool_blocks, int G);
bool attn_krot_map(CUtensorMap* m, const __half* krot, int n_pages, int G);
// Bytes of the rotated-K scratch for n_pages pages.
size_t attention_krot_bytes(int n_pages, int G);
// CTAs of the tensor-core attention for a plan of n_items items (the grid barrier's count).
int attention_tc_grid(int n_items);
// For callers holding fp32 pre-RoPE a.q (kernel-level calls): writes the rotated fp16 copy
// into q16 ([T][H][128], 16-byte aligned), zeroes the grid-barrier counter *sync (8 bytes of
// device memory) and sets a.q16, a.krot (attention_krot_bytes of a.n_pages pages, 16-byte
// aligned, filled by the attention kernel), the barrier and the maps (V pool of pool_blocks
// blocks).
pic_status attention_prepare_tc(AttnArgs& a, int T, int pool_blocks, __half* q16, __half* krot,
                                unsigned long long* sync, cudaStream_t st);
void plan_attention(const AttnPlanInput& in, std::vector<AttnItem>& items, std::vector<AttnCombine>& combines,
                    int& n_parts);
size_t attention_part_bytes(int n_parts, int rep, int D);

// ------------------------------------------------------------------ dynamic selection (k_select.cu)
// One request of a dynamic-selection pass: its query rows [row0, row0 + lq) of the pass's
// layer-0 QKV rows, its n_tok prompt tokens (scores [tok0, tok0 + n_tok)), its prompt pages
// [page0, page0 + n_pages) of the pass's page arrays, the n_pick positions it keeps
// (chosen[out0, out0 + n_pick), ascending), its blocks of 64 keys over the prompt and the
// query (from kb0) and over the prompt alone (from pkb0), and its logits [lq][H][n_tok + lq]
// from float lg0 of the logits scratch.
struct SelectReq {
  int row0, lq, n_tok, tok0, page0, n_pages, n_pick, out0, kb0, pkb0, lg0;
};
constexpr int kSelectReqInts = sizeof(SelectReq) / sizeof(int);
constexpr int kSelectKeyBlock = 64;   // keys per block of the scoring kernels
struct SelectArgs {
  const SelectReq* reqs;    // device, ascending row0, tok0, kb0, pkb0
  int n_reqs, n_rows, n_tok, H, G;
  int n_kb, n_pkb;          // key blocks over prompt + query keys, over prompt keys (all requests)
  const float* qkv;         // [n_rows][(H + 2G) D] fp32 layer-0 projections of the query rows
  const void* k_layer0;     // layer 0 of the K pool [blocks][G][16][D], model dtype, pre-RoPE
  const int* page_block;    // pages of every request's prompt, position order
  const int* page_pos;      // position of each page's row 0 within its request's prompt
  const int* page_len;
  const float2* rope_cs;    // [positions][D/2]
  float* qrot;              // scratch [n_rows][H][D]
  float* logits;            // scratch, the requests' logits (SelectReq::lg0)
  float* ml;                // scratch [n_rows][H][2]: max, 1 / sum
  float* scores;            // [n_tok] out
  int* chosen;              // out
};
// Scores every prompt token and writes each request's chosen positions (5 launches).
pic_status launch_select(const SelectArgs& a, int D, int dtype, cudaStream_t st);

void rope_table_host(int n_pos, int D, double base, std::vector<float2>& out);

}  // namespace pic
