// tcgen05 tensor-core GEMM for the projections of the selected rows (bf16 in, fp32 out).
//
//   Y[t][n] += sum_k W[n][k] * X[t][k]        (Y fp32, accumulated in place)
//
// The link step multiplies a few hundred selected rows by large weight matrices, so
// the weights take the MMA's M side (128 rows per CTA) and the token rows its N side
// (up to 256 per tile): one weight tile is streamed from HBM exactly once per token
// tile. Operands are staged by TMA (128-byte swizzle, K-major) through a multi-stage
// mbarrier ring; one thread issues tcgen05.mma with the fp32 accumulator in TMEM; all
// four warps drain TMEM with tcgen05.ld into a shared-memory tile that one TMA bulk
// reduce-add folds into Y. Split-K spreads the weight stream over every SM; the splits
// meet in Y through those reductions, so no partial slabs are written or re-read, and a
// projection that feeds the residual stream adds straight into it.
//
// Every mbarrier wait is bounded (~2 s of GPU time). On expiry the kernel raises a
// device flag, stops issuing work, waits (bounded) for the copies and MMAs it started,
// frees its TMEM and returns; the host reports PIC_ERR_DEVICE_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "pic_internal.h"

namespace pic {

namespace {

constexpr int BM = 128;          // weight rows per MMA (M); a CTA tile holds 1 or 2 of these
constexpr int BK = 64;           // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;       // K per tcgen05.mma (kind::f16)
constexpr int A_HALF_BYTES = BM * BK * 2;
constexpr int kThreads = 128;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ int g_tc_timeout = 0;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity; false (and the device flag) on expiry.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 255u) == 0 && gtimer() - t0 > kWaitLimitNs) {
      atomicExch(&g_tc_timeout, 1);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);   // start address
  // leading byte offset: unused for K-major tiles whose K extent fits one swizzle row
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset between 8-row atoms
  d |= (uint64_t)1 << 46;                     // descriptor version
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

struct TcParams {
  int N, K, T;
  int BN;            // token rows per tile (multiple of 16, <= 256)
  int stages;
  int kb_per_split;  // k-blocks of BK per split
  int nkb;           // total k-blocks
  uint32_t tmem_cols;
};

// MH = 128-row weight halves per CTA tile. Both halves share the staged activation
// tile, so MH = 2 halves the activation bytes read from L2 per weight byte streamed.
template <int MH>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                   const __grid_constant__ CUtensorMap map_y, const TcParams p) {
  constexpr int A_STAGE_BYTES = MH * A_HALF_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = A_STAGE_BYTES + p.BN * BK * 2;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.stages * stage_bytes);
  // bars[0..S): full, bars[S..2S): empty, bars[2S]: accumulator ready
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * p.stages + 1);
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * BM * MH, t0 = blockIdx.y * p.BN, split = blockIdx.z;
  const int kb0 = split * p.kb_per_split;
  const int nk = min(p.nkb - kb0, p.kb_per_split);
  const uint32_t acc_bar = smem_u32(bars + 2 * p.stages);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < 2 * p.stages + 1; ++i) mbar_init(smem_u32(bars + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(p.tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    asm volatile("tcgen05.fence::before_thread_sync;");
  }
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    uint64_t pol_w, pol_x;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % p.stages;
      const uint32_t ph = (kb / p.stages) & 1;
      if (!mbar_wait(smem_u32(bars + p.stages + st), ph ^ 1)) {
        s_abort = 1;
        break;
      }
      const uint32_t full = smem_u32(bars + st);
      const uint32_t a_dst = smem_u32(smem + st * stage_bytes);
      const uint32_t b_dst = a_dst + A_STAGE_BYTES;
      mbar_expect_tx(full, stage_bytes);
      const int kx = (kb0 + kb) * BK;
#pragma unroll
      for (int hf = 0; hf < MH; ++hf) tma_load_2d(a_dst + hf * A_HALF_BYTES, &map_w, kx, m0 + hf * BM, full, pol_w);
      tma_load_2d(b_dst, &map_x, kx, t0, full, pol_x);
      issued = kb + 1;
    }
    // copies still in flight must land before this CTA's shared memory is released
    for (int kb = max(0, issued - p.stages); kb < issued; ++kb)
      if (!mbar_wait(smem_u32(bars + kb % p.stages), (kb / p.stages) & 1)) break;
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    const uint32_t idesc = idesc_bf16(BM, p.BN);
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % p.stages;
      if (s_abort || !mbar_wait(smem_u32(bars + st), (kb / p.stages) & 1)) {
        s_abort = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;");
      const uint32_t a_base = smem_u32(smem + st * stage_bytes);
      const uint32_t b_base = a_base + A_STAGE_BYTES;
#pragma unroll
      for (int k = 0; k < BK / UMMA_K; ++k) {
        const uint64_t bd = smem_desc_sw128(b_base + k * UMMA_K * 2);
#pragma unroll
        for (int hf = 0; hf < MH; ++hf) {
          const uint64_t ad = smem_desc_sw128(a_base + hf * A_HALF_BYTES + k * UMMA_K * 2);
          umma_bf16(tmem + hf * p.BN, ad, bd, idesc, (kb | k) != 0);
        }
      }
      umma_commit(smem_u32(bars + p.stages + st));  // stage free once these MMAs retire
    }
    umma_commit(acc_bar);  // accumulator complete (or abandoned) once every MMA retires
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> shared tile [BN][128] fp32 -> TMA reduce-add into Y
  bool ok = mbar_wait(acc_bar, 0);
  ok = __syncthreads_and(ok) && !s_abort;  // block-uniform; warps reconverged for .sync.aligned loads
  asm volatile("tcgen05.fence::after_thread_sync;");
  if (ok) {
    // every staged operand has been consumed by the MMAs, so the ring's memory is free
    float* S = reinterpret_cast<float*>(smem);
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int nl = warp * 32 + lane;
#pragma unroll
    for (int hf = 0; hf < MH; ++hf) {
      for (int c = 0; c < p.BN; c += 16) {
        float v[16];
        tmem_ld16(lane_base + hf * p.BN + c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) S[(c + j) * BM + nl] = v[j];
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      if (threadIdx.x == 0) {
        asm volatile(
            "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                reinterpret_cast<uint64_t>(&map_y)),
            "r"(m0 + hf * BM), "r"(t0), "r"(smem_u32(S))
            : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // tile read out before it is reused
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols));
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// fp32 [rows][cols] destination of the bulk reduce-add; box = 128 columns x box_rows rows
bool make_map_f32(CUtensorMap* m, void* base, int rows, int cols, int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {(cuuint32_t)BM, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int pick_bn(int T) {
  if (T >= 256) return 256;
  return std::max(16, (T + 15) / 16 * 16);
}

}  // namespace

bool tc_gemm_supported(int N, int K, int T) { return N >= BM && N % BM == 0 && K >= BK && K % BK == 0 && T >= 1; }

// Two weight halves per CTA when the shape allows (N multiple of 256, at most 256 token
// rows per tile so both fp32 accumulators fit the 512 TMEM columns).
int pick_mh(int N, int T) { return (N % (2 * BM) == 0) ? 2 : 1; }

int tc_gemm_splits(int N, int K, int T, int num_sms, int max_splits) {
  const int BN = pick_bn(T);
  const long long tiles = (long long)(N / (BM * pick_mh(N, T))) * ((T + BN - 1) / BN);
  const int nkb = K / BK;
  const int smax = std::max(1, std::min({max_splits, nkb / 4, 16}));
  const double epi = 2.0;  // epilogue cost in k-block units
  int best = 1;
  double best_t = 1e30;
  for (int s = 1; s <= smax; ++s) {
    const int kps = (nkb + s - 1) / s;
    const int real_s = (nkb + kps - 1) / kps;
    const long long ctas = tiles * real_s;
    const long long waves = (ctas + num_sms - 1) / num_sms;
    const double t = (double)waves * (kps + epi);
    if (t < best_t - 1e-9) {
      best_t = t;
      best = real_s;
    }
  }
  return best;
}

pic_status tc_gemm_run(const void* W, const void* X, float* Y, int N, int K, int T, int splits, cudaStream_t st) {
  if (!tc_gemm_supported(N, K, T)) return fail(PIC_ERR_UNSUPPORTED, "tcgen05 gemm: unsupported shape");
  if (((uintptr_t)W | (uintptr_t)X | (uintptr_t)Y) % 16)
    return fail(PIC_ERR_INVALID_ARG, "tcgen05 gemm: operands not 16-byte aligned");
  TcParams p{};
  p.N = N;
  p.K = K;
  p.T = T;
  p.BN = pick_bn(T);
  p.nkb = K / BK;
  splits = std::max(1, std::min(splits, p.nkb));
  p.kb_per_split = (p.nkb + splits - 1) / splits;
  const int real_splits = (p.nkb + p.kb_per_split - 1) / p.kb_per_split;
  if (real_splits != splits) return fail(PIC_ERR_INVALID_ARG, "tcgen05 gemm: split count leaves an empty split");
  const int mh = pick_mh(N, T);
  const int stage_bytes = mh * A_HALF_BYTES + p.BN * BK * 2;
  const int budget = 227 * 1024 - 2048;  // opt-in limit minus alignment slack, barriers and static smem
  p.stages = std::max(2, std::min(8, budget / stage_bytes));
  p.tmem_cols = 32;
  while ((int)p.tmem_cols < mh * p.BN) p.tmem_cols <<= 1;
  if ((size_t)p.stages * stage_bytes < (size_t)p.BN * BM * 4)
    return fail(PIC_ERR_UNSUPPORTED, "tcgen05 gemm: staging tile does not fit the pipeline memory");
  CUtensorMap mw, mx, my;
  if (!make_map(&mw, W, N, K, BM) || !make_map(&mx, X, T, K, p.BN) || !make_map_f32(&my, Y, T, N, p.BN))
    return fail(PIC_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  const size_t smem = 1024 + (size_t)p.stages * stage_bytes + (2 * p.stages + 2) * 8;
  // raise the kernel's dynamic shared-memory limit to what this launch needs (once per size, per device)
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t attr_smem[2][64] = {};
  auto kern = mh == 2 ? tc_gemm_kernel<2> : tc_gemm_kernel<1>;
  if (dev < 0 || dev >= 64 || attr_smem[mh - 1][dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("tcgen05 gemm attribute: ") + cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) attr_smem[mh - 1][dev] = smem;
  }
  dim3 grid(N / (BM * mh), (T + p.BN - 1) / p.BN, splits);
  kern<<<grid, kThreads, smem, st>>>(mw, mx, my, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("tcgen05 gemm launch: ") + cudaGetErrorString(e));
  return PIC_OK;
}

pic_status tc_check_timeout() {
  int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_timeout, sizeof(int));
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("timeout flag: ") + cudaGetErrorString(e));
  if (v) {
    cudaMemcpyToSymbol(g_tc_timeout, &zero, sizeof(int));
    return fail(PIC_ERR_DEVICE_TIMEOUT, "a tensor-core kernel gave up a bounded wait");
  }
  return PIC_OK;
}

}  // namespace pic
