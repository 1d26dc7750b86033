// SIMT FFMA GEMM: Y[t][n] += sum_k X[t][k] * W[n][k], fp32 accumulation; K may be split
// over CTAs, whose sums meet in Y through atomic adds.
// Used for fp32 models (tcgen05 has no plain-fp32 kind) and for shapes the tensor-core
// kernel does not take. 64x64 output tile per CTA, 4x4 per thread, K in steps of 16.
#include "pic_internal.h"

namespace pic {

namespace {

constexpr int BN = 64, BT = 64, BK = 16;

template <typename TW, typename TX>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const TW* __restrict__ W, const TX* __restrict__ X,
                                                        float* __restrict__ Y, int N, int K, int T,
                                                        int k_per_split) {
  __shared__ float Ws[BK][BN + 4];
  __shared__ float Xs[BK][BT + 4];
  const int n0 = blockIdx.x * BN, t0 = blockIdx.y * BT, s = blockIdx.z;
  const int kb = s * k_per_split, ke = min(K, kb + k_per_split);
  const int tid = threadIdx.x;
  const int tn = (tid % 16) * 4, tt = (tid / 16) * 4;
  float acc[4][4] = {};
  for (int k0 = kb; k0 < ke; k0 += BK) {
    for (int i = tid; i < BN * BK; i += 256) {
      const int r = i / BK, c = i % BK;
      const int n = n0 + r, k = k0 + c;
      Ws[c][r] = (n < N && k < ke) ? to_f<TW>(W[(size_t)n * K + k]) : 0.f;
      const int t = t0 + r;
      Xs[c][r] = (t < T && k < ke) ? to_f<TX>(X[(size_t)t * K + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < BK; ++c) {
      float a[4], b[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a[j] = Ws[c][tn + j];
        b[j] = Xs[c][tt + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(b[i], a[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + tt + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tn + j;
      if (n < N) atomicAdd(Y + (size_t)t * N + n, acc[i][j]);
    }
  }
}

}  // namespace

void launch_gemm_simt(int w_dtype, bool x_half, const void* W, const void* X, float* Y, int N, int K, int T,
                      int splits, cudaStream_t st) {
  if (T <= 0 || N <= 0) return;
  int kps = (K + splits - 1) / splits;
  kps = (kps + BK - 1) / BK * BK;
  dim3 grid((N + BN - 1) / BN, (T + BT - 1) / BT, splits);
  if (w_dtype == PIC_BF16 && x_half)
    gemm_simt_kernel<__nv_bfloat16, __half><<<grid, 256, 0, st>>>((const __nv_bfloat16*)W, (const __half*)X, Y, N, K,
                                                                  T, kps);
  else if (w_dtype == PIC_BF16)
    gemm_simt_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)W,
                                                                         (const __nv_bfloat16*)X, Y, N, K, T, kps);
  else
    gemm_simt_kernel<float, float><<<grid, 256, 0, st>>>((const float*)W, (const float*)X, Y, N, K, T, kps);
}

}  // namespace pic
