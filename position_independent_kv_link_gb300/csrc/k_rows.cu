// Row-wise kernels of the decoder around the GEMMs and attention: embedding gather +
// RMSNorm, the QKV epilogue (q out, pre-RoPE K/V scattered into page slots), RMSNorm of the
// residual stream, SwiGLU, block copies for request-private pages, KV import. All are
// memory-bound; float4 accesses over rows.
#include <algorithm>
#include <type_traits>

#include "pic_internal.h"

namespace pic {

namespace {

constexpr int kRowThreads = 256;

// fp16 range guard. For bf16 models the tensor cores take fp16 operands: the activations these
// kernels write (normed rows, SwiGLU output, the rotated and scaled q) and, inside attention, K
// rotated by RoPE and V. A value outside fp16's finite range (|x| > 65504, or NaN) would become
// inf there without notice, so the kernels that write those values set this word instead;
// pic_sync reports it as PIC_ERR_RANGE. Stored K is checked against 46000: a rotation mixes two
// components and can grow one by up to sqrt(2) (65504 / sqrt(2) = 46319).
__device__ unsigned int g_range_flag = 0;
constexpr float kF16Max = 65504.f;
constexpr float kKRotMax = 46000.f;
__device__ __forceinline__ bool outside(float x, float lim) { return !(fabsf(x) <= lim); }
__device__ __forceinline__ bool outside4(float4 v, float lim) {
  return outside(v.x, lim) | outside(v.y, lim) | outside(v.z, lim) | outside(v.w, lim);
}
__device__ __forceinline__ void flag_range(bool bad) {
  if (bad) atomicOr(&g_range_flag, 1u);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x < 32) {
    s = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (l == 0) red[0] = s;
  }
  __syncthreads();
  s = red[0];
  __syncthreads();
  return s;
}

// h = E[tok]; x = rmsnorm(h) * g.  Row cached in dynamic shared memory (fp32).
template <typename T, typename A>
__global__ void embed_norm_kernel(int d, const T* __restrict__ E, const int* __restrict__ tok,
                                  const float* __restrict__ gain, float eps, float* __restrict__ h,
                                  A* __restrict__ x) {
  pdl_enter();
  extern __shared__ float row[];
  __shared__ float red[32];
  const int t = blockIdx.x;
  const T* e = E + (size_t)tok[t] * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float v = to_f<T>(e[i]);
    row[i] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / d + eps);
  bool bad = false;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    h[(size_t)t * d + i] = row[i];
    const float y = row[i] * r * gain[i];
    if constexpr (std::is_same<A, __half>::value) bad |= outside(y, kF16Max);
    x[(size_t)t * d + i] = from_f<A>(y);
  }
  flag_range(bad);
}

template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) {
  *reinterpret_cast<float4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = u;
}

template <>
__device__ __forceinline__ void store4<__half>(__half* dst, float4 v) {
  flag_range(outside4(v, kF16Max));
  __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = u;
}

// 4 accumulator floats (the accumulators are zeroed before their GEMM, not cleared here:
// clearing behind the read costs about as much again as the read)
__device__ __forceinline__ float4 take4(const float* __restrict__ acc, size_t off) {
  return *reinterpret_cast<const float4*>(acc + off);
}

// QKV epilogue: q -> [T][H*D] fp32; pre-RoPE k, v -> their page slot of this layer. The
// accumulator [T][N] is only read. grid (T, ceil(N / 1024)); a thread owns 4
// consecutive columns (one head).
// Dims i..i+3 and i+64..i+67 (i < 64) of one 128-dim q head: rotate-half RoPE at the angles of
// one table row, times `scale`, rounded once to fp16.
__device__ __forceinline__ void rope_q16_store(float4 a, float4 b, const float2* __restrict__ cs_row, int i, float scale,
                                               __half* __restrict__ dst) {
  const float x1[4] = {a.x, a.y, a.z, a.w}, x2[4] = {b.x, b.y, b.z, b.w};
  float y1[4], y2[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 c = cs_row[i + e];
    y1[e] = (x1[e] * c.x - x2[e] * c.y) * scale;
    y2[e] = (x2[e] * c.x + x1[e] * c.y) * scale;
  }
  store4<__half>(dst + i, make_float4(y1[0], y1[1], y1[2], y1[3]));
  store4<__half>(dst + 64 + i, make_float4(y2[0], y2[1], y2[2], y2[3]));
}

template <typename T>
__global__ void qkv_epilogue_kernel(int H, int G, int D, const float* __restrict__ acc, float* __restrict__ q,
                                    const int* __restrict__ slot, T* __restrict__ kl, T* __restrict__ vl,
                                    const int* __restrict__ pos, const float2* __restrict__ rope_cs,
                                    __half* __restrict__ q16) {
  pdl_enter();
  const int t = blockIdx.x;
  const int N = (H + 2 * G) * D;
  const int n = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (n >= N) return;
  if (q16 && n < H * D) {   // rotated fp16 q: the thread of dims i < 64 also takes dims i + 64
    const int i = n % D;
    if (i >= 64) return;
    const size_t base = (size_t)t * N + n;
    const float4 a = take4(acc, base), b = take4(acc, base + 64);
    rope_q16_store(a, b, rope_cs + (size_t)pos[t] * 64, i, kQ16Scale, q16 + (size_t)t * H * D + (n - i));
    return;
  }
  const float4 v = take4(acc, (size_t)t * N + n);
  if (n < H * D) {
    store4<float>(q + (size_t)t * H * D + n, v);
  } else {
    const int s_ = slot[t];
    const int blk = s_ / kBlock, r = s_ % kBlock;
    const int m = n - H * D;
    const int kv = m / (G * D);          // 0: K, 1: V
    const int g = (m % (G * D)) / D, i = m % D;
    T* dst = kv == 0 ? kl : vl;
    if constexpr (std::is_same<T, __nv_bfloat16>::value) flag_range(outside4(v, kv == 0 ? kKRotMax : kF16Max));
    store4<T>(dst + (((size_t)blk * G + g) * kBlock + r) * D + i, v);
  }
}

// y = RMSNorm(h[t]) * gain (the projection GEMMs have already added into h). Not final:
// x[t] = y in the model dtype. Final: hidden_out[out_row[t]] = y (fp32) and
// lm_x[lg_row[t]] = y (model dtype) where those indices are >= 0.
template <typename T>
__global__ void __launch_bounds__(512) rmsnorm_rows_kernel(int d, const float* __restrict__ h,
                                                           const float* __restrict__ gain, float eps,
                                                           T* __restrict__ x, int final_layer,
                                                           const int* __restrict__ out_row,
                                                           float* __restrict__ hidden_out,
                                                           const int* __restrict__ lg_row, T* __restrict__ lm_x) {
  pdl_enter();
  __shared__ float red[32];
  const int t = blockIdx.x;
  const float* hr = h + (size_t)t * d;
  float ss = 0.f;
  for (int i = threadIdx.x * 4; i < d; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(hr + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / d + eps);
  const int o = final_layer ? out_row[t] : -1, lg = final_layer ? lg_row[t] : -1;
  if (final_layer && o < 0 && lg < 0) return;
  for (int i = threadIdx.x * 4; i < d; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(hr + i);
    const float4 g = *reinterpret_cast<const float4*>(gain + i);
    const float4 y = make_float4(v.x * r * g.x, v.y * r * g.y, v.z * r * g.z, v.w * r * g.w);
    if (!final_layer) {
      store4<T>(x + (size_t)t * d + i, y);
    } else {
      if (o >= 0) *reinterpret_cast<float4*>(hidden_out + (size_t)o * d + i) = y;
      if (lg >= 0) store4<T>(lm_x + (size_t)lg * d + i, y);
    }
  }
}

// act = silu(gate) * up from the accumulator [T][2F] (gate columns, then up columns), which
// is only read. grid (T, ceil(F / 1024)); 4 outputs per thread.
template <typename T>
__global__ void swiglu_kernel(int F, const float* __restrict__ acc, T* __restrict__ act) {
  pdl_enter();
  const int t = blockIdx.x;
  const int j = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (j >= F) return;
  const size_t N = 2 * (size_t)F;
  const float4 a = take4(acc, (size_t)t * N + j);
  const float4 b = take4(acc, (size_t)t * N + F + j);
  const float4 y = make_float4(a.x / (1.f + __expf(-a.x)) * b.x, a.y / (1.f + __expf(-a.y)) * b.y,
                               a.z / (1.f + __expf(-a.z)) * b.z, a.w / (1.f + __expf(-a.w)) * b.w);
  store4<T>(act + (size_t)t * F + j, y);
}

// p[0..n) = 0: 16-byte stores where p is 16-byte aligned, the rest one float at a time
__device__ __forceinline__ void zero_range(float* __restrict__ p, size_t n, size_t i0, size_t step) {
  const size_t n4 = ((uintptr_t)p % 16 == 0) ? n / 4 : 0;
  for (size_t i = i0; i < n4; i += step) reinterpret_cast<float4*>(p)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (size_t i = 4 * n4 + i0; i < n; i += step) p[i] = 0.f;
}
__global__ void zero_kernel(float* __restrict__ p, size_t n, float* __restrict__ p2, size_t n2) {
  pdl_enter();
  const size_t i0 = blockIdx.x * (size_t)blockDim.x + threadIdx.x, step = (size_t)gridDim.x * blockDim.x;
  zero_range(p, n, i0, step);
  if (p2) zero_range(p2, n2, i0, step);
}

// grid: (pairs, layers, 2 pools); 16-byte copies of one block of one layer.
__global__ void copy_blocks_kernel(const int* __restrict__ pairs, int num_blocks_total, size_t block_bytes,
                                   char* __restrict__ kp, char* __restrict__ vp) {
  pdl_enter();
  const int i = blockIdx.x, l = blockIdx.y;
  char* pool = blockIdx.z == 0 ? kp : vp;
  const size_t layer_off = (size_t)l * num_blocks_total * block_bytes;
  const int4* src = reinterpret_cast<const int4*>(pool + layer_off + (size_t)pairs[2 * i] * block_bytes);
  int4* dst = reinterpret_cast<int4*>(pool + layer_off + (size_t)pairs[2 * i + 1] * block_bytes);
  for (size_t j = threadIdx.x; j < block_bytes / 16; j += blockDim.x) dst[j] = src[j];
}

// grid: (n tokens, layers); copies K and V rows of one token into its page slot.
template <typename T>
__global__ void import_kv_kernel(int n, int G, int D, const T* __restrict__ ks, const T* __restrict__ vs,
                                 const int* __restrict__ blocks, int num_blocks_total, T* __restrict__ kp,
                                 T* __restrict__ vp) {
  const int t = blockIdx.x, l = blockIdx.y;
  const int blk = blocks[t / kBlock], r = t % kBlock;
  const size_t src = ((size_t)l * n + t) * G * D;
  for (int j = threadIdx.x; j < G * D; j += blockDim.x) {
    const int g = j / D, i = j % D;
    const size_t dst = ((((size_t)l * num_blocks_total + blk) * G + g) * kBlock + r) * D + i;
    const T k = ks[src + j], v = vs[src + j];
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
      flag_range(outside(to_f<T>(k), kKRotMax) | outside(to_f<T>(v), kF16Max));
    kp[dst] = k;
    vp[dst] = v;
  }
}

}  // namespace

pic_status rows_check_range() {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_range_flag, sizeof(v));
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("range flag: ") + cudaGetErrorString(e));
  if (v) {
    cudaMemcpyToSymbol(g_range_flag, &zero, sizeof(zero));
    return fail(PIC_ERR_RANGE, "a value bound for an fp16 tensor-core operand was outside fp16's range (|x| > 65504, "
                               "or > 46000 for stored K, or NaN); the outputs since the last pic_sync are invalid");
  }
  return PIC_OK;
}

void rows_raise_range() {
  const unsigned one = 1;
  cudaMemcpyToSymbol(g_range_flag, &one, sizeof(one));
}

void launch_embed_norm(int dtype, int T, int d, const void* embed, const int* tok, const float* gain, float eps,
                       float* h, void* x, cudaStream_t st) {
  if (T <= 0) return;
  const size_t sm = d * sizeof(float);
  if (dtype == PIC_BF16)
    launch_dependent(embed_norm_kernel<__nv_bfloat16, __half>, dim3(T), dim3(kRowThreads), sm, st, d, (const __nv_bfloat16*)embed, tok, gain,
                                                                         eps, h, (__half*)x);
  else
    launch_dependent(embed_norm_kernel<float, float>, dim3(T), dim3(kRowThreads), sm, st, d, (const float*)embed, tok, gain, eps, h,
                                                                (float*)x);
}

void launch_qkv_epilogue(int dtype, int T, int H, int G, int D, float* acc, float* q, const int* slot, void* k_layer,
                         void* v_layer, const int* pos, const float2* rope_cs, __half* q16, cudaStream_t st) {
  if (T <= 0) return;
  const int N = (H + 2 * G) * D;
  dim3 grid(T, (N / 4 + kRowThreads - 1) / kRowThreads);
  if (dtype == PIC_BF16)
    launch_dependent(qkv_epilogue_kernel<__nv_bfloat16>, grid, dim3(kRowThreads), 0, st,
        H, G, D, acc, q, slot, (__nv_bfloat16*)k_layer, (__nv_bfloat16*)v_layer, pos, rope_cs, q16);
  else
    launch_dependent(qkv_epilogue_kernel<float>, grid, dim3(kRowThreads), 0, st, H, G, D, acc, q, slot, (float*)k_layer,
                                                             (float*)v_layer, pos, rope_cs, nullptr);
}

namespace {
__global__ void rope_q16_kernel(int H, const float* __restrict__ q, const int* __restrict__ pos,
                                const float2* __restrict__ rope_cs, __half* __restrict__ q16) {
  const int t = blockIdx.x;
  const int j = blockIdx.y * blockDim.x + threadIdx.x;   // (head, i / 4) with i < 64
  if (j >= H * 16) return;
  const int h = j / 16, i = (j % 16) * 4;
  const float* src = q + ((size_t)t * H + h) * 128;
  rope_q16_store(*reinterpret_cast<const float4*>(src + i), *reinterpret_cast<const float4*>(src + 64 + i),
                 rope_cs + (size_t)pos[t] * 64, i, kQ16Scale, q16 + ((size_t)t * H + h) * 128);
}
}  // namespace

void launch_rope_q16(int T, int H, const float* q, const int* pos, const float2* rope_cs, __half* q16,
                     cudaStream_t st) {
  if (T <= 0) return;
  rope_q16_kernel<<<dim3(T, (H * 16 + 255) / 256), 256, 0, st>>>(H, q, pos, rope_cs, q16);
}

void launch_rmsnorm_rows(int dtype, int T, int d, const float* h, const float* gain, float eps, void* x,
                         bool final_layer, const int* out_row, float* hidden_out, const int* lg_row, void* lm_x,
                         cudaStream_t st) {
  if (T <= 0) return;
  const int thr = std::min(512, std::max(128, (d / 4 + 31) / 32 * 32));
  if (dtype == PIC_BF16)
    launch_dependent(rmsnorm_rows_kernel<__half>, dim3(T), dim3(thr), 0, st, d, h, gain, eps, (__half*)x, (int)final_layer, out_row, hidden_out,
                                                   lg_row, (__half*)lm_x);
  else
    launch_dependent(rmsnorm_rows_kernel<float>, dim3(T), dim3(thr), 0, st, d, h, gain, eps, (float*)x, (int)final_layer, out_row, hidden_out,
                                                  lg_row, (float*)lm_x);
}

void launch_swiglu(int dtype, int T, int F, float* acc, void* act, cudaStream_t st) {
  if (T <= 0) return;
  dim3 grid(T, (F / 4 + kRowThreads - 1) / kRowThreads);
  if (dtype == PIC_BF16)
    launch_dependent(swiglu_kernel<__half>, grid, dim3(kRowThreads), 0, st, F, (const float*)acc, (__half*)act);
  else
    launch_dependent(swiglu_kernel<float>, grid, dim3(kRowThreads), 0, st, F, (const float*)acc, (float*)act);
}

void launch_zero(float* p, size_t n, cudaStream_t st, float* p2, size_t n2) {
  if (n == 0 && n2 == 0) return;
  const unsigned blocks = (unsigned)std::min<size_t>(4096, (std::max(n, n2) / 4 + 255) / 256 + 1);
  launch_dependent(zero_kernel, dim3(blocks), dim3(256), 0, st, p, n, p2, n2);
}

void launch_copy_blocks(int n_pairs, const int* pairs, int n_layers, int num_blocks_total, size_t block_bytes,
                        void* k_pool, void* v_pool, cudaStream_t st) {
  if (n_pairs <= 0) return;
  dim3 grid(n_pairs, n_layers, 2);
  launch_dependent(copy_blocks_kernel, grid, dim3(256), 0, st, pairs, num_blocks_total, block_bytes, (char*)k_pool,
                   (char*)v_pool);
}

void launch_import_kv(int dtype, int n_layers, int n, int G, int D, const void* k_src, const void* v_src,
                      const int* blocks, int num_blocks_total, void* k_pool, void* v_pool, cudaStream_t st) {
  if (n <= 0) return;
  dim3 grid(n, n_layers);
  if (dtype == PIC_BF16)
    import_kv_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(n, G, D, (const __nv_bfloat16*)k_src,
                                                          (const __nv_bfloat16*)v_src, blocks, num_blocks_total,
                                                          (__nv_bfloat16*)k_pool, (__nv_bfloat16*)v_pool);
  else
    import_kv_kernel<float><<<grid, 256, 0, st>>>(n, G, D, (const float*)k_src, (const float*)v_src, blocks,
                                                  num_blocks_total, (float*)k_pool, (float*)v_pool);
}

}  // namespace pic
