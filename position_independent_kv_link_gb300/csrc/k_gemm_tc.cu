// tcgen05 tensor-core GEMM for the projections of the selected rows (bf16 in, fp32 out).
//
//   Y[t][n] += sum_k W[n][k] * X[t][k]        (Y fp32, accumulated in place)
//
// The link step multiplies a few hundred selected rows by large weight matrices: the
// weights take the MMA's M side (128 rows per tile) and the token rows its N side (up
// to 256 per tile), so each weight tile is streamed from HBM once per token tile. Every
// weight k-block (16 KB) brings the token tile's k-block (up to 32 KB, from L2) into the SM
// with it; from 1024 token rows on (compute-bound, 4+ token tiles) the packed layout takes two
// weight tiles per activation tile (256 weight rows: two M = 128 MMAs per K step into two
// accumulators that fill the TMEM, one accumulator set).
//
// Persistent, stream-K, warp-specialized. The grid has one CTA per SM; the linear space
// of (tile, 64-wide k-block) work is cut into equal contiguous ranges, one per CTA, so
// every SM streams the same number of weight bytes. A CTA walks its range as segments
// (maximal runs inside one tile). Each segment accumulates in one of two TMEM buffers
// (one set of two halves for 256-row tiles) and is folded into Y by TMA bulk reduce-adds,
// so segments of the same tile that land on different CTAs meet in Y with no fix-up pass,
// and (128-row tiles) the drain of one segment overlaps the MMAs of the next.
//
//   warp 0     TMA producer: weight tile(s) + activation tile of each k-block into one stage
//   warp 1     MMA issuer (one thread): tcgen05.mma kind::f16, fp32 accumulators in TMEM,
//              one tcgen05.commit per k-block to free its stage
//   warp 2     TMEM owner (alloc/dealloc)
//   warps 3-   epilogue, four warps per 128-row half: tcgen05.ld -> 16-row shared tile ->
//              cp.reduce.async.bulk add
//
// For the model's fixed weights it is launched as a programmatic dependent of the previous
// kernel in the stream: the producer fills the first pipeline stages with weight tiles (which
// no kernel of the forward writes) while that kernel finishes, then waits for it
// (griddepcontrol.wait) before the first activation load; the epilogue waits the same way
// before its first reduce-add. Without that launch attribute the waits return at once.
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

constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BK = 64;           // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;       // K per tcgen05.mma (kind::f16)
constexpr int A_STAGE = BM * BK * 2;   // 16 KB
constexpr int EPI_ROWS = 16;     // token rows per reduce-add tile
constexpr int EPI_COLS = 32;     // weight rows per reduce-add tile: one epilogue warp's TMEM lane quarter
constexpr int EPI_BYTES = EPI_ROWS * BM * 4;  // 8 KB: the four warps' tiles, double buffered
// MW weight tiles of 128 rows share each k-block's activation tile (MW = 2: two M = 128 MMAs
// per K step into two accumulators). Warps: producer, MMA issuer, TMEM owner, then four
// epilogue warps per 128-row half. With MW = 2 the two accumulators of up to 256 columns fill
// the TMEM, so there is one accumulator set instead of two alternating ones.
template <int MW>
struct Wide {
  static constexpr int kWarps = 3 + 4 * MW;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kAcc = MW == 1 ? 2 : 1;   // accumulator sets
};
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ int g_tc_timeout = 0;
__device__ int g_pack_range = 0;   // a packed weight was outside fp16's finite range (or NaN)

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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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

// 1-D bulk copy of a contiguous global range into shared memory, completing on `bar`
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1024 B apart.
// (The leading byte offset is unused for K-major tiles whose K extent fits one swizzle row.)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset between 8-row atoms
  d |= (uint64_t)1 << 46;                     // descriptor version
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: A and B both bf16 (fmt 1) or both fp16 (fmt 0),
// both K-major, fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, uint32_t fmt) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
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

// tcgen05.ld of 16 columns without waiting; tmem_wait16 on the same registers before using them
// (the registers are operands of the wait, so no use can be scheduled ahead of it)
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// named barrier of the N epilogue threads
template <int N>
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// same barrier with an AND over the N epilogue threads: all of them take the same branch
template <int N>
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(N)
      : "memory");
  return r != 0;
}

struct TcParams {
  const uint8_t* w_packed;  // PACKED: [N/128][K/64] tiles of 16 KB in their shared-memory image
  int N, K, T;
  int BN;            // token rows per tile (multiple of 16, <= 256)
  int S;             // pipeline stages (one k-block of weights + activations each)
  int nkb;           // k-blocks per tile
  int m_tiles;       // weight-row tiles (of 128 MW rows)
  int total;         // tiles * nkb work units (< 2^31, checked on the host)
  uint32_t ab_fmt;   // operand format of both A and B: 1 = bf16, 0 = fp16
  uint32_t tmem_cols;
  // Y starts at zero inside the kernel (no separate clearing pass): the CTA whose range holds a
  // tile's first k-block zeroes the tile's part of Y and then sets tile_ready[tile] = epoch;
  // every reduce-add into a tile waits for that. Null: Y is accumulated into as it is.
  int* tile_ready;
  uint32_t epoch;
  float* Y;          // raw Y [T][N] (for the zeroing)
};

// The order a CTA walks its range [lo, hi). Every segment is drained (a full tile of reduce-adds)
// whatever its length; with one accumulator set (256-row weight tiles) a drain holds up the next
// segment's MMAs, and a range that ends with a segment shorter than the one it starts with would
// finish with two drains back to back. Such a range is walked from the start m of its last
// segment: [m, hi), then [lo, m), so the short segment's drain comes first, under the longer
// segments' weight loads (measured: 32-request batch 80.0 -> 74.5 ms, full recompute 81.6 ->
// 75.7 ms). With two accumulator sets the plain order is kept: there the reorder measured slower
// (k = 32 7.07 -> 7.51 ms), as CTAs a token tile apart no longer reach a weight band together and
// share it through L2. The producer, the MMA issuer and the epilogue walk the same order.
struct Walk {
  int a0, b0, a1, b1;   // units [a0, b0), then [a1, b1)
};
__device__ __forceinline__ Walk range_walk(int lo, int hi, int nkb, bool reorder) {
  const int m = max(lo, (hi - 1) / nkb * nkb);          // first unit of the last segment
  const int first_end = min(hi, (lo / nkb + 1) * nkb);  // end of the first segment
  if (reorder && m > lo && hi - m < first_end - lo) return Walk{m, hi, lo, m};
  return Walk{lo, hi, hi, hi};
}
// the i-th unit of the walk
__device__ __forceinline__ int walk_unit(const Walk& w, int i) {
  const int n0 = w.b0 - w.a0;
  return i < n0 ? w.a0 + i : w.a1 + (i - n0);
}

// Segment walk shared by the MMA issuer and the epilogue: [g, end) inside one tile.
struct Seg {
  int g, end;
  int tile;
};
__device__ __forceinline__ bool next_seg(Seg& s, int hi, int nkb) {
  s.g = s.end;
  if (s.g >= hi) return false;
  s.tile = s.g / nkb;
  s.end = min(hi, (s.tile + 1) * nkb);
  return true;
}

// PACKED: weight tiles come from the pre-swizzled tile copy by one contiguous 16 KB bulk
// copy each (sequential DRAM pages); otherwise by a 2-D tensor copy of the [N][K] matrix.
template <bool PACKED, int MW>
__global__ void __launch_bounds__(Wide<MW>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                   const __grid_constant__ CUtensorMap map_y, const TcParams p) {
  static_assert(PACKED || MW == 1, "wide tiles take the packed weights");
  constexpr int kAcc = Wide<MW>::kAcc;
  constexpr int kEpi = 128 * MW;   // epilogue threads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_stage = p.BN * BK * 2;
  const int stage = MW * A_STAGE + b_stage;                   // one k-block: MW weight tiles, then activation tile
  uint8_t* ring = smem;
  uint8_t* epi = ring + p.S * stage;                          // [4 MW warps][2][16][32] fp32
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + 2 * MW * EPI_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = full + p.S;
  uint64_t* acc_full = empty + p.S;        // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lo = (int)((long long)p.total * blockIdx.x / gridDim.x);
  const int hi = (int)((long long)p.total * (blockIdx.x + 1) / gridDim.x);
  const Walk wk = range_walk(lo, hi, p.nkb, kAcc == 1);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < p.S; ++i) {
      mbar_init(smem_u32(full + i), 1);
      mbar_init(smem_u32(empty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(acc_full + i), 1);
      mbar_init(smem_u32(acc_empty + i), 4 * MW);   // one arrival per epilogue warp
    }
    mbar_init(smem_u32(mma_done), 1);
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
    // ---------------- TMA producer: weight tile (HBM stream, evicted first from L2) and
    // activation tile (small, reused by every weight tile, kept in L2) of each k-block, in the
    // range's walk order.
    uint64_t pol_w, pol_x;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
    int st = 0, issued = 0;
    uint32_t ph = 0;
    const int n_units = hi - lo;
    // weights of the first stages before the previous kernel has finished, then its outputs
    const int pre = min(p.S, n_units);
    for (int i = 0; i < pre; ++i) {
      const int u = walk_unit(wk, i), kb = u % p.nkb, mt = (u / p.nkb) % p.m_tiles;
      const uint32_t fb = smem_u32(full + i), dst = smem_u32(ring + i * stage);
      mbar_expect_tx(fb, stage);
      if (PACKED)
#pragma unroll
        for (int h = 0; h < MW; ++h)
          bulk_load(dst + h * A_STAGE, p.w_packed + ((size_t)(mt * MW + h) * p.nkb + kb) * A_STAGE, A_STAGE, fb,
                    pol_w);
      else
        tma_load_2d(dst, &map_w, kb * BK, mt * BM, fb, pol_w);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");   // the next kernel may launch and wait for us
    for (int i = 0; i < pre; ++i) {
      const int u = walk_unit(wk, i), kb = u % p.nkb, tt = (u / p.nkb) / p.m_tiles;
      tma_load_2d(smem_u32(ring + i * stage) + MW * A_STAGE, &map_x, kb * BK, tt * p.BN, smem_u32(full + i), pol_x);
      ++issued;
      if (++st == p.S) {
        st = 0;
        ph ^= 1;
      }
    }
    // (k-block, weight tile, token tile) of each unit advance incrementally: no division in the
    // loop but at the walk's one jump between its two ranges
    const int n0 = wk.b0 - wk.a0;
    int kb = 0, mt = 0, tt = 0;
    auto locate = [&](int u) {
      kb = u % p.nkb;
      const int tile = u / p.nkb;
      mt = tile % p.m_tiles;
      tt = tile / p.m_tiles;
    };
    if (pre < n_units) locate(walk_unit(wk, pre));
    for (int i = pre; i < n_units; ++i) {
      if (s_abort || !mbar_wait(smem_u32(empty + st), ph ^ 1)) {
        s_abort = 1;
        break;
      }
      const uint32_t fb = smem_u32(full + st);
      const uint32_t dst = smem_u32(ring + st * stage);
      mbar_expect_tx(fb, stage);
      if (PACKED)
#pragma unroll
        for (int h = 0; h < MW; ++h)
          bulk_load(dst + h * A_STAGE, p.w_packed + ((size_t)(mt * MW + h) * p.nkb + kb) * A_STAGE, A_STAGE, fb, pol_w);
      else
        tma_load_2d(dst, &map_w, kb * BK, mt * BM, fb, pol_w);
      tma_load_2d(dst + MW * A_STAGE, &map_x, kb * BK, tt * p.BN, fb, pol_x);
      ++issued;
      if (++st == p.S) {
        st = 0;
        ph ^= 1;
      }
      if (i + 1 == n0) {
        locate(wk.a1);
      } else if (++kb == p.nkb) {
        kb = 0;
        if (++mt == p.m_tiles) {
          mt = 0;
          ++tt;
        }
      }
    }
    for (int j = max(0, issued - p.S); j < issued; ++j)   // land in-flight copies before exit
      if (!mbar_wait(smem_u32(full + j % p.S), (uint32_t)((j / p.S) & 1))) break;
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: one commit per k-block releases its stage
    const uint32_t idesc = idesc_f16kind(BM, p.BN, p.ab_fmt);
    int s = 0, st = 0;
    uint32_t ph = 0;
    bool stop = false;
    for (int r = 0; r < 2 && !stop && !s_abort; ++r) {
    Seg sg{0, r ? wk.a1 : wk.a0, 0};
    const int seg_end = r ? wk.b1 : wk.b0;
    while (!stop && next_seg(sg, seg_end, p.nkb)) {
      const int ab = kAcc == 2 ? (s & 1) : 0;
      const uint32_t use = kAcc == 2 ? (uint32_t)(s >> 1) : (uint32_t)s;   // earlier uses of this accumulator set
      if (s_abort || !mbar_wait(smem_u32(acc_empty + ab), (use & 1) ^ 1)) {
        s_abort = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;");
      const uint32_t d_tmem = tmem + ab * MW * p.BN;   // half h at + h BN
      for (int g = sg.g; g < sg.end; ++g) {
        if (s_abort || !mbar_wait(smem_u32(full + st), ph)) {
          s_abort = 1;
          stop = true;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t a_base = smem_u32(ring + st * stage);
        const uint32_t b_base = a_base + MW * A_STAGE;
#pragma unroll
        for (int h = 0; h < MW; ++h)
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            umma_bf16(d_tmem + h * p.BN, smem_desc_sw128(a_base + h * A_STAGE + k * UMMA_K * 2),
                      smem_desc_sw128(b_base + k * UMMA_K * 2), idesc, (g != sg.g || k != 0) ? 1u : 0u);
        umma_commit(smem_u32(empty + st));  // the stage is free once these MMAs retire
        if (++st == p.S) {
          st = 0;
          ph ^= 1;
        }
      }
      if (!stop) umma_commit(smem_u32(acc_full + ab));
      ++s;
    }
    }
    umma_commit(smem_u32(mma_done));          // fires once every MMA of this CTA has retired
    mbar_wait(smem_u32(mma_done), 0);
  } else if (warp >= 3) {
    // ---------------- epilogue: TMEM -> [16 tokens][32 rows] fp32 tiles -> bulk reduce-add into Y
    const int e = warp - 3;                    // epilogue warp: 128-row half e / 4
    const int hw = e >> 2;
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const bool leader = (warp == 3 && lane == 0);
    float* stg = reinterpret_cast<float*>(epi);
    asm volatile("griddepcontrol.wait;" ::: "memory");   // Y is written by earlier kernels
    if (p.tile_ready) {
      // zero the tiles whose first k-block is in this CTA's range: 32 MW threads per row of 128 MW
      // columns (16-byte stores), 4 rows per pass; then publish them
      const int ep = threadIdx.x - 3 * 32;   // 0 .. 128 MW - 1
      const int t_tiles_bn = p.BN;
      for (int tile = (lo + p.nkb - 1) / p.nkb; tile * p.nkb < hi; ++tile) {
        const int m0 = (tile % p.m_tiles) * BM * MW, t0 = (tile / p.m_tiles) * t_tiles_bn;
        const int rows = min(t_tiles_bn, p.T - t0);
        for (int rr = ep / (32 * MW); rr < rows; rr += 4)
          reinterpret_cast<float4*>(p.Y + (size_t)(t0 + rr) * p.N + m0)[ep % (32 * MW)] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __threadfence();
      epi_bar<kEpi>();
      if (leader)
        for (int tile = (lo + p.nkb - 1) / p.nkb; tile * p.nkb < hi; ++tile)
          asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.tile_ready + tile), "r"(p.epoch) : "memory");
    }
    int s = 0, buf = 0;
    bool quit = false;   // the same in all epilogue threads (set after epi_all)
    for (int r = 0; r < 2 && !quit; ++r) {
    Seg sg{0, r ? wk.a1 : wk.a0, 0};
    const int seg_end = r ? wk.b1 : wk.b0;
    while (next_seg(sg, seg_end, p.nkb)) {
      const int ab = kAcc == 2 ? (s & 1) : 0;
      const uint32_t use = kAcc == 2 ? (uint32_t)(s >> 1) : (uint32_t)s;
      bool ok = !s_abort && mbar_wait(smem_u32(acc_full + ab), use & 1);
      ok = epi_all<kEpi>(ok);
      if (!ok) {
        s_abort = 1;
        quit = true;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;");
      const int m0 = (sg.tile % p.m_tiles) * BM * MW + hw * BM, t0 = (sg.tile / p.m_tiles) * p.BN;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (ab * MW + hw) * p.BN;
      if (p.tile_ready && lane == 0) {
        // the tile's zeroing (by the CTA holding its first k-block) has landed
        const unsigned long long w0 = gtimer();
        for (uint32_t i = 0;; ++i) {
          uint32_t v;
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.tile_ready + sg.tile) : "memory");
          if (v == p.epoch) break;
          if ((i & 63) == 63 && (s_abort || gtimer() - w0 > kWaitLimitNs)) {
            atomicExch(&g_tc_timeout, 1);
            s_abort = 1;
            break;
          }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");   // the reduce-adds come after the zeroes
      }
      // Each warp drains its own 32 weight rows on its own: 16 token columns per step from TMEM
      // (the next step's load in flight while this one is staged) into its [16][32] fp32 tile,
      // bulk reduce-added into Y by the warp's first lane, two tiles alternating.
      float* W = stg + e * (2 * EPI_ROWS * EPI_COLS);
      uint32_t cur[16], nxt[16];
      tmem_ld16_async(taddr, cur);
      tmem_wait16(cur);
      for (int c = 0; c < p.BN; c += EPI_ROWS) {
        if (c + EPI_ROWS < p.BN) tmem_ld16_async(taddr + c + EPI_ROWS, nxt);
        float* S = W + buf * (EPI_ROWS * EPI_COLS);
#pragma unroll
        for (int j = 0; j < 16; ++j) S[j * EPI_COLS + lane] = __uint_as_float(cur[j]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          if (t0 + c < p.T)
            asm volatile(
                "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                    reinterpret_cast<uint64_t>(&map_y)),
                "r"(m0 + q * EPI_COLS), "r"(t0 + c), "r"(smem_u32(S))
                : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");  // the other tile is free again
        }
        __syncwarp();
        buf ^= 1;
        if (c + EPI_ROWS < p.BN) {
          tmem_wait16(nxt);
#pragma unroll
          for (int j = 0; j < 16; ++j) cur[j] = nxt[j];
        }
      }
      // the MMAs of the segment after next may overwrite this accumulator
      asm volatile("tcgen05.fence::before_thread_sync;");
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(acc_empty + ab));
      ++s;
    }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols));
}

// [N][K] bf16 -> [N/128][K/64] fp16 tiles of 128 rows x 64 k, each stored exactly as a
// 128-byte-swizzled K-major shared-memory tile (16-byte chunk j of row r at slot j ^ (r % 8)).
__global__ void pack_sw128_kernel(const uint4* __restrict__ W, uint4* __restrict__ P, int K, int nkb) {
  const int tile = blockIdx.x;            // mt * nkb + kb
  const int mt = tile / nkb, kb = tile % nkb;
  for (int i = threadIdx.x; i < BM * 8; i += blockDim.x) {
    const int r = i / 8, j = i % 8;
    const uint4 v = W[((size_t)(mt * BM + r) * K + kb * BK) / 8 + j];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint4 o;
    __half2* h = reinterpret_cast<__half2*>(&o);
    bool bad = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(b[e]);
      bad |= !(fabsf(f.x) <= 65504.f) | !(fabsf(f.y) <= 65504.f);
      h[e] = __float22half2_rn(f);
    }
    if (bad) atomicExch(&g_pack_range, 1);
    P[(size_t)tile * (A_STAGE / 16) + r * 8 + (j ^ (r & 7))] = o;
  }
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

// fp32 [rows][cols] destination of the bulk reduce-add; box = EPI_COLS columns x EPI_ROWS rows
bool make_map_f32(CUtensorMap* m, void* base, int rows, int cols) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {(cuuint32_t)EPI_COLS, (cuuint32_t)EPI_ROWS};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 16-bit K-major operand [rows][K] (bf16 or fp16); box = 64 K x box_rows rows, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows, bool f16 = false) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Token rows per tile: the fewest tiles of at most 256 rows, of equal height rounded up to 16
// (1632 rows: 7 tiles of 240 rather than 6 of 256 and one of 96, which would pad the MMAs by 10 %)
int pick_bn(int T) {
  const int n = std::max(1, (T + 255) / 256);
  return std::max(16, ((T + n - 1) / n + 15) / 16 * 16);
}

// Weight tiles per activation tile: 2 (256 weight rows) for the packed layout from 1024 token
// rows on, when N holds whole 256-row tiles. There the GEMM is compute-bound over 4 or more
// token tiles, and each 16 KB weight k-block would bring a 32 KB activation k-block into the SM
// with it: measured on the 8B link shapes, 5120-5184 rows run 6-9 % faster this way and 2048
// rows (a compile call) 5 %, while 224 and 384 rows run 9 % and 6 % slower (their single
// accumulator set serialises each drain with the next segment).
int pick_mw(bool packed, int N, int T) { return packed && N % (2 * BM) == 0 && T >= 1024 ? 2 : 1; }

int device_sms() {
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = n > 0 ? n : 148;
  }
  return sms[dev];
}

}  // namespace

bool tc_gemm_supported(int N, int K, int T) { return N >= BM && N % BM == 0 && K >= BK && K % BK == 0 && T >= 1; }

namespace {

pic_status tc_gemm_launch(const void* W, bool packed, const void* X, float* Y, int N, int K, int T, cudaStream_t st,
                          bool early_weights, int* tile_ready, uint32_t epoch) {
  if (!tc_gemm_supported(N, K, T)) return fail(PIC_ERR_UNSUPPORTED, "tcgen05 gemm: unsupported shape");
  if (((uintptr_t)W | (uintptr_t)X | (uintptr_t)Y) % 16)
    return fail(PIC_ERR_INVALID_ARG, "tcgen05 gemm: operands not 16-byte aligned");
  TcParams p{};
  p.w_packed = packed ? static_cast<const uint8_t*>(W) : nullptr;
  p.tile_ready = tile_ready;
  p.epoch = epoch;
  p.Y = Y;
  p.ab_fmt = packed ? 0u : 1u;   // the packed copy is fp16 (X too); the plain layout is bf16
  p.N = N;
  p.K = K;
  p.T = T;
  p.BN = pick_bn(T);
  p.nkb = K / BK;
  const int wide = pick_mw(packed, N, T);   // weight tiles per activation tile
  p.m_tiles = N / (BM * wide);
  const long long tiles = (long long)p.m_tiles * ((T + p.BN - 1) / p.BN);
  if (tiles * p.nkb >= (1LL << 31)) return fail(PIC_ERR_UNSUPPORTED, "tcgen05 gemm: shape too large");
  p.total = (int)(tiles * p.nkb);
  const int b_stage = p.BN * BK * 2;
  // shared memory: as many stages as fit next to the epilogue tiles and the barriers
  const int budget = 227 * 1024 - 1024 - 2 * wide * EPI_BYTES - 512;
  p.S = std::min(12, budget / (wide * A_STAGE + b_stage));
  if (p.S < 2) return fail(PIC_ERR_UNSUPPORTED, "tcgen05 gemm: pipeline does not fit shared memory");
  p.tmem_cols = 32;   // two accumulator sets of one BN-column tile, or one set of two (wide = 2)
  while ((int)p.tmem_cols < 2 * p.BN) p.tmem_cols <<= 1;
  CUtensorMap mw, mx, my;
  std::memset(&mw, 0, sizeof(mw));
  if ((!packed && !make_map(&mw, W, N, K, BM)) || !make_map(&mx, X, T, K, p.BN, packed) ||
      !make_map_f32(&my, Y, T, N))
    return fail(PIC_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  const size_t smem =
      1024 + (size_t)p.S * (wide * A_STAGE + b_stage) + 2 * wide * EPI_BYTES + (2 * p.S + 6) * 8 + 16;
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t attr_smem[3][64] = {};
  const int variant = packed ? wide : 0;
  auto kern = !packed ? tc_gemm_kernel<false, 1> : wide == 2 ? tc_gemm_kernel<true, 2> : tc_gemm_kernel<true, 1>;
  const int threads = wide == 2 ? Wide<2>::kThreads : Wide<1>::kThreads;
  if (dev < 0 || dev >= 64 || attr_smem[variant][dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("tcgen05 gemm attribute: ") + cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) attr_smem[variant][dev] = smem;
  }
  const int grid = std::min(device_sms(), p.total);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = early_weights ? 1 : 0;
  cudaLaunchKernelEx(&cfg, kern, mw, mx, my, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("tcgen05 gemm launch: ") + cudaGetErrorString(e));
  return PIC_OK;
}

}  // namespace

pic_status tc_gemm_run(const void* W, const void* X, float* Y, int N, int K, int T, cudaStream_t st) {
  return tc_gemm_launch(W, false, X, Y, N, K, T, st, false, nullptr, 0);
}

pic_status tc_gemm_run_packed(const void* Wp, const void* X, float* Y, int N, int K, int T, cudaStream_t st,
                              bool early_weights, int* tile_ready, uint32_t epoch) {
  return tc_gemm_launch(Wp, true, X, Y, N, K, T, st, early_weights, tile_ready, epoch);
}

size_t tc_gemm_tiles(int N, int T) {   // of the packed layout's launch
  return (size_t)(N / (BM * pick_mw(true, N, T))) * ((T + pick_bn(T) - 1) / pick_bn(T));
}

pic_status tc_pack_weight(const void* W, void* out, int N, int K, cudaStream_t st) {
  if (!tc_gemm_supported(N, K, 1)) return fail(PIC_ERR_UNSUPPORTED, "pack: N % 128 and K % 64 must be 0");
  if (((uintptr_t)W | (uintptr_t)out) % 16) return fail(PIC_ERR_INVALID_ARG, "pack: pointers not 16-byte aligned");
  const int nkb = K / BK;
  pack_sw128_kernel<<<(N / BM) * nkb, 256, 0, st>>>((const uint4*)W, (uint4*)out, K, nkb);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("pack launch: ") + cudaGetErrorString(e));
  return PIC_OK;
}

pic_status tc_check_pack_range() {
  int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_pack_range, sizeof(int));
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("pack range flag: ") + cudaGetErrorString(e));
  if (v) {
    cudaMemcpyToSymbol(g_pack_range, &zero, sizeof(int));
    return fail(PIC_ERR_RANGE, "a projection weight is outside fp16's range (|w| > 65504 or NaN): it cannot be packed "
                               "as an fp16 tensor-core operand");
  }
  return PIC_OK;
}

void tc_raise_timeout() {
  const int one = 1;
  cudaMemcpyToSymbol(g_tc_timeout, &one, sizeof(int));
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
