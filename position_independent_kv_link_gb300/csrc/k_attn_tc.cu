// tcgen05 paged attention with fused RoPE for bf16 KV, head_dim 128, 4 query heads per KV head.
//
// One CTA = one work item: up to 32 consecutive query rows of one sequence x the 4 query
// heads that share KV head g x a run of pages. The 32 rows x 4 heads are exactly one
// M = 128 MMA tile (row m = head * 32 + row), so each 64-key tile of K and V is staged
// once and read by the tensor cores once for all of them.
//
//   warps 0-3  softmax: thread = one MMA row = one TMEM lane. Reads its row of S from
//              TMEM, masks keys after its position (and padding), keeps a running
//              reference maximum, writes P = 2^(S - ref) as fp16 into shared memory and
//              sums it. O in TMEM is rescaled only when the maximum grows by more than
//              2^8 (P stays <= 256, safe in fp16); the same reference is used for the
//              sum, so the final O / l is exact softmax.
//   warps 4-7  transform: cp.async of the raw bf16 K/V pages one tile ahead, then K is
//              rotated by RoPE at each key's absolute position (MEPIC abstract: K is kept
//              without positional encoding and RoPE is fused into attention) and V is
//              transposed, both to fp16 in the 128-byte-swizzled K-major layout of the MMA
//              operands. cos/sin(p theta) is composed from the table row of the page start
//              and the row of the offset inside the page.
//   warp 8     TMEM owner; one thread issues S = Q K^T (M128 N64 K128, into one of two
//              TMEM buffers) and O += P V (M128 N128 K64) with tcgen05.mma kind::f16.
// Page metadata is cached in shared memory in windows of 512 pages. Every mbarrier wait is
// bounded; on expiry the CTA raises the device timeout flag and winds down.
#include <climits>

#include "pic_internal.h"

namespace pic {

bool tc_attention_supported(int dtype, int D, int rep);
void launch_attention_tc(const AttnArgs& a, cudaStream_t st);

namespace {

constexpr int D = 128;
constexpr int REP = 4;
constexpr int RB = 32;                    // query rows per item
constexpr int KT = 64;                    // keys per tile
constexpr int WIN = 512;
constexpr int kThreads = 9 * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescale = 8.f;           // rescale O when the row max grows by more than 2^8
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// shared memory map (bytes from a 1024-aligned base)
constexpr int OFF_Q = 0;                       // 2 halves x [128 rows][128 B]        32 KB
constexpr int OFF_K = OFF_Q + 32768;           // [2 buf][2 halves][64 rows][128 B]    32 KB
constexpr int OFF_VT = OFF_K + 32768;          // [2 buf][128 dims][128 B = 64 keys]   32 KB
constexpr int OFF_P = OFF_VT + 32768;          // [2 buf][128 rows][128 B = 64 keys]   32 KB
constexpr int OFF_RAW = OFF_P + 32768;         // [2 buf][K 16 KB | V 16 KB] bf16      64 KB
constexpr int OFF_LO = OFF_RAW + 65536;        // float2 [16][64]                       8 KB
constexpr int OFF_PG = OFF_LO + 8192;          // float2 [2][4][64]                     4 KB
constexpr int OFF_META = OFF_PG + 4096;        // int [3][WIN]                          6 KB
constexpr int OFF_TM = OFF_META + 3 * WIN * 4; // int [2][4][2] (page start, valid rows)
constexpr int OFF_POS = OFF_TM + 64;           // int [2][KT]
constexpr int OFF_BAR = OFF_POS + 2 * KT * 4;  // mbarriers
constexpr int N_BARS = 12;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16;

__device__ int g_attn_timeout = 0;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
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
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 255u) == 0 && gtimer() - t0 > kWaitLimitNs) {
      atomicExch(&g_attn_timeout, 1);
      return false;
    }
  }
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// named barrier of the four transform warps, with an AND so that all take the same branch
__device__ __forceinline__ bool tr_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 2, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void tr_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// 16-byte chunk c (0..7) of row r of a [rows][128 B] tile, 128-byte swizzle (UMMA K-major)
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }
// 16-byte chunk c (0..15) of row r of a [rows][256 B] raw tile, XOR-swizzled
__device__ __forceinline__ uint32_t swz256(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16, A and B fp16 K-major, D fp32, M x N
__device__ __forceinline__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
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
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// rotate dims (8c..8c+7) and (64+8c..) by the composed angle, times `scale`, to fp16
__device__ __forceinline__ void rope8(const float* v1, const float* v2, const float2* hi, const float2* lo, float scale,
                                      uint4& y1, uint4& y2) {
  __half o1[8], o2[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float2 H2 = hi[e], L2 = lo[e];
    const float cs = H2.x * L2.x - H2.y * L2.y, sn = H2.y * L2.x + H2.x * L2.y;
    o1[e] = __float2half_rn((v1[e] * cs - v2[e] * sn) * scale);
    o2[e] = __float2half_rn((v2[e] * cs + v1[e] * sn) * scale);
  }
  y1 = *reinterpret_cast<uint4*>(o1);
  y2 = *reinterpret_cast<uint4*>(o2);
}
__device__ __forceinline__ void bf8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(b[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float2* sLo = reinterpret_cast<float2*>(sm + OFF_LO);
  float2* sPg = reinterpret_cast<float2*>(sm + OFF_PG);
  int* sBlk = reinterpret_cast<int*>(sm + OFF_META);
  int* sPp = sBlk + WIN;
  int* sPl = sPp + WIN;
  int* sTm = reinterpret_cast<int*>(sm + OFF_TM);   // [buf][page][start, valid rows]
  int* sPos = reinterpret_cast<int*>(sm + OFF_POS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  // [0,2) kv_full  [2,4) s_full  [4,6) s_free  [6,8) p_full  [8,10) pv_done  [10] mma_done
  const uint32_t b_kvfull = smem_u32(bars), b_sfull = smem_u32(bars + 2), b_sfree = smem_u32(bars + 4),
                 b_pfull = smem_u32(bars + 6), b_pvdone = smem_u32(bars + 8), b_mmadone = smem_u32(bars + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + N_BARS);
  __shared__ volatile int s_abort;

  const AttnItem it = a.items[blockIdx.x];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npages = it.page1 - it.page0;
  const int ntiles = (npages + 3) / 4;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_kvfull + 8 * i, 4);
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_sfree + 8 * i, 4);
      mbar_init(b_pfull + 8 * i, 4);
      mbar_init(b_pvdone + 8 * i, 1);
    }
    mbar_init(b_mmadone, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(256));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  for (int i = tid; i < 16 * 64; i += kThreads) sLo[i] = a.rope_cs[i];
  __syncthreads();

  // ---- Q tile: row m = head * 32 + row, rotated at the row's position, scaled into log2 units
  const float qscale = rsqrtf((float)D) * kLog2e;
  for (int i = tid; i < 128 * 8; i += kThreads) {
    const int m = i / 8, c = i % 8, hh = m / RB, r = m % RB;
    uint4 y1 = make_uint4(0, 0, 0, 0), y2 = y1;
    if (r < it.nrows) {
      const int t = it.row0 + r, h = it.g * REP + hh, p = a.q_pos[t];
      const float* src = a.q + ((size_t)t * a.H + h) * D;
      float v1[8], v2[8];
      *reinterpret_cast<float4*>(v1) = *reinterpret_cast<const float4*>(src + 8 * c);
      *reinterpret_cast<float4*>(v1 + 4) = *reinterpret_cast<const float4*>(src + 8 * c + 4);
      *reinterpret_cast<float4*>(v2) = *reinterpret_cast<const float4*>(src + 64 + 8 * c);
      *reinterpret_cast<float4*>(v2 + 4) = *reinterpret_cast<const float4*>(src + 64 + 8 * c + 4);
      rope8(v1, v2, a.rope_cs + (size_t)(p & ~15) * 64 + 8 * c, sLo + (p & 15) * 64 + 8 * c, qscale, y1, y2);
    }
    *reinterpret_cast<uint4*>(sm + OFF_Q + sw128(m, c)) = y1;
    *reinterpret_cast<uint4*>(sm + OFF_Q + 16384 + sw128(m, c)) = y2;
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;   // O: columns [0,128); S buffer b: [128 + 64 b, 192 + 64 b)

  if (warp < 4) {
    // =============================== softmax warps
    const int hh = warp, r = lane, m = hh * RB + r;
    const int qp = r < it.nrows ? a.q_pos[it.row0 + r] : -1;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float mref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int b = j & 1, u = j >> 1;
      // kv_full of the same tile also orders this thread after the transform's key positions
      ok = __all_sync(0xffffffffu,
                      !s_abort && mbar_wait(b_sfull + 8 * b, u & 1) && mbar_wait(b_kvfull + 8 * b, u & 1));
      if (!ok) break;
      fence_after();
      float s[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld16(trow + 128 + 64 * b + 16 * c, s + 16 * c);
      tmem_wait_ld();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sfree + 8 * b);
      const int* kp = sPos + b * KT;
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        if (kp[i] > qp) s[i] = -INFINITY;
        mx = fmaxf(mx, s[i]);
      }
      // new reference when the maximum grows by more than 2^8 (or for the first keys seen)
      const bool grow = mx > mref + kRescale || (mref == -INFINITY && mx > -INFINITY);
      const float mnew = grow ? mx : mref;
      const float scale = (grow && mref != -INFINITY) ? exp2f(mref - mnew) : 1.f;
      if (__any_sync(0xffffffffu, scale != 1.f)) {
        // O holds the sums of the tiles before: rescale it once PV of the previous tile is done
        if (!mbar_wait(b_pvdone + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1)) {
          s_abort = 1;
          ok = false;
        }
        if (!__all_sync(0xffffffffu, ok)) break;
        fence_after();
        for (int c = 0; c < 128; c += 16) {
          float o[16];
          tmem_ld16(trow + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] *= scale;
          tmem_st16(trow + c, o);
        }
        tmem_wait_st();
        fence_before();
      }
      l *= scale;
      mref = mnew;
      // P = 2^(S - ref) in fp16 into the operand tile; P of tile j - 2 must have been consumed
      if (j >= 2 && !mbar_wait(b_pvdone + 8 * b, (u - 1) & 1)) {
        s_abort = 1;
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      uint8_t* prow = sm + OFF_P + b * 16384;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        __half hv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float p = mref == -INFINITY ? 0.f : exp2f(s[8 * c + e] - mref);
          rs += p;
          hv[e] = __float2half_rn(p);
        }
        *reinterpret_cast<uint4*>(prow + sw128(m, c)) = *reinterpret_cast<uint4*>(hv);
      }
      l += rs;
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull + 8 * b);
    }
    // ---- output: O / l (or the unnormalized partial with its reference max and sum)
    if (ok && ntiles > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(b_pvdone + 8 * ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1));
      if (!ok) s_abort = 1;
    }
    if (ok) {
      fence_after();
      const int h = it.g * REP + hh;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      for (int c = 0; c < 128; c += 16) {
        float o[16];
        if (ntiles > 0) {
          tmem_ld16(trow + c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = 0.f;
        }
        if (it.part < 0) {
          if (r < it.nrows) {
            __half hv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) hv[e] = __float2half_rn(o[e] * inv);
            __half* dst = (__half*)a.out + ((size_t)(it.row0 + r) * a.H + h) * D + c;
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<uint4*>(hv);
            *reinterpret_cast<uint4*>(dst + 8) = *reinterpret_cast<uint4*>(hv + 8);
          }
        } else {
          float* dst = a.part_o + (((size_t)it.part * kAttnPartRows + r) * REP + hh) * D + c;
#pragma unroll
          for (int e = 0; e < 16; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        }
      }
      if (it.part >= 0) {
        const size_t pi = ((size_t)it.part * kAttnPartRows + r) * REP + hh;
        a.part_ml[pi * 2] = mref;
        a.part_ml[pi * 2 + 1] = l;
      }
    }
  } else if (warp < 8) {
    // =============================== transform warps: raw pages -> fp16 K (rotated) and V^T
    const int tt = tid - 128;
    const __nv_bfloat16* Kl = (const __nv_bfloat16*)a.k_layer;
    const __nv_bfloat16* Vl = (const __nv_bfloat16*)a.v_layer;
    int win = -1;
    auto issue = [&](int tile) {
      const int b = tile & 1;
      const int w1 = (tile * 4 / WIN) * WIN;
      if (w1 != win) {   // same decision in every transform thread
        tr_bar();
        win = w1;
        for (int i = tt; i < WIN; i += 128) {
          const int pg = it.page0 + win + i;
          if (pg < it.page1) {
            sBlk[i] = a.page_block[pg];
            sPp[i] = a.page_pos[pg];
            sPl[i] = a.page_len[pg];
          }
        }
        tr_bar();
      }
      const int pbase = tile * 4 - win;
      if (tt < 4) {
        const bool in = tile * 4 + tt < npages;
        sTm[(b * 4 + tt) * 2] = in ? sPp[pbase + tt] : 0;
        sTm[(b * 4 + tt) * 2 + 1] = in ? sPl[pbase + tt] : 0;
      }
      uint8_t* raw = sm + OFF_RAW + b * 32768;
      for (int task = tt; task < KT * 16; task += 128) {
        const int key = task / 16, c = task % 16, pg = key / 16, rr = key % 16;
        if (tile * 4 + pg < npages && rr < sPl[pbase + pg]) {
          const size_t src = (((size_t)sBlk[pbase + pg] * a.G + it.g) * kBlock + rr) * D + 8 * c;
          cp_async16(smem_u32(raw + swz256(key, c)), Kl + src);
          cp_async16(smem_u32(raw + 16384 + swz256(key, c)), Vl + src);
        }
      }
      {  // RoPE rows of the tile's four page starts
        const int pg = tt / 32, c = tt % 32;
        if (tile * 4 + pg < npages)
          cp_async16(smem_u32(sPg + (b * 4 + pg) * 64) + c * 16, a.rope_cs + (size_t)sPp[pbase + pg] * 64 + c * 2);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    bool ok = true;
    if (ntiles > 0) issue(0);
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1, u = j >> 1;
      tr_bar();   // every thread is done reading the raw buffer the next issue overwrites
      if (j + 1 < ntiles) {
        issue(j + 1);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      // operand buffer b is free once PV of tile j - 2 has retired
      ok = tr_all(!s_abort && (j < 2 || mbar_wait(b_pvdone + 8 * b, (u - 1) & 1)));
      if (!ok) {
        s_abort = 1;
        break;
      }
      const uint8_t* raw = sm + OFF_RAW + b * 32768;
      uint8_t* kt = sm + OFF_K + b * 16384;
      uint8_t* vt = sm + OFF_VT + b * 16384;
      // K: rotate (dims c and c + 64 together)
      for (int task = tt; task < KT * 8; task += 128) {
        const int key = task / 8, c = task % 8, pg = key / 16, rr = key % 16;
        const bool valid = rr < sTm[(b * 4 + pg) * 2 + 1];
        uint4 y1 = make_uint4(0, 0, 0, 0), y2 = y1;
        if (valid) {
          float v1[8], v2[8];
          bf8_to_f32(*reinterpret_cast<const uint4*>(raw + swz256(key, c)), v1);
          bf8_to_f32(*reinterpret_cast<const uint4*>(raw + swz256(key, c + 8)), v2);
          rope8(v1, v2, sPg + (b * 4 + pg) * 64 + 8 * c, sLo + rr * 64 + 8 * c, 1.f, y1, y2);
        }
        *reinterpret_cast<uint4*>(kt + sw128(key, c)) = y1;
        *reinterpret_cast<uint4*>(kt + 8192 + sw128(key, c)) = y2;
        if (c == 0) sPos[b * KT + key] = valid ? sTm[(b * 4 + pg) * 2] + rr : INT_MAX;
      }
      // V: transpose to [dim][key] fp16 (the K-major operand of O += P V)
      for (int task = tt; task < KT * 16; task += 128) {
        const int key = task % KT, c = task / KT, pg = key / 16, rr = key % 16;
        const bool valid = rr < sTm[(b * 4 + pg) * 2 + 1];
        float v[8];
        if (valid) {
          bf8_to_f32(*reinterpret_cast<const uint4*>(raw + 16384 + swz256(key, c)), v);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int d = 8 * c + e;
          *reinterpret_cast<__half*>(vt + sw128(d, key / 8) + (key % 8) * 2) = __float2half_rn(v[e]);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_kvfull + 8 * b);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (lane == 0) {
    // =============================== MMA issuer
    const uint32_t id_s = idesc_f16(128, KT), id_pv = idesc_f16(128, D);
    const uint32_t qa = smem_u32(sm + OFF_Q);
    auto issue_s = [&](int j) -> bool {
      const int b = j & 1, u = j >> 1;
      if (s_abort || !mbar_wait(b_kvfull + 8 * b, u & 1)) return false;
      if (j >= 2 && !mbar_wait(b_sfree + 8 * b, (u - 1) & 1)) return false;
      fence_after();
      const uint32_t kb = smem_u32(sm + OFF_K + b * 16384);
#pragma unroll
      for (int k = 0; k < 8; ++k) {   // K dimension 128 = 2 halves x 4 steps of 16
        const uint32_t off = (k & 3) * 32;
        umma(tmem + 128 + 64 * b, desc_sw128(qa + (k >> 2) * 16384 + off), desc_sw128(kb + (k >> 2) * 8192 + off),
             id_s, k != 0);
      }
      umma_commit(b_sfull + 8 * b);
      return true;
    };
    bool ok = ntiles == 0 || issue_s(0);
    for (int j = 0; j < ntiles && ok; ++j) {
      if (j + 1 < ntiles && !issue_s(j + 1)) {
        ok = false;
        break;
      }
      const int b = j & 1, u = j >> 1;
      if (s_abort || !mbar_wait(b_pfull + 8 * b, u & 1)) {
        ok = false;
        break;
      }
      fence_after();
      const uint32_t pa = smem_u32(sm + OFF_P + b * 16384), vb = smem_u32(sm + OFF_VT + b * 16384);
#pragma unroll
      for (int k = 0; k < 4; ++k)   // K dimension 64 keys = 4 steps of 16
        umma(tmem, desc_sw128(pa + k * 32), desc_sw128(vb + k * 32), id_pv, (j | k) != 0);
      umma_commit(b_pvdone + 8 * b);
    }
    if (!ok) s_abort = 1;
    umma_commit(b_mmadone);   // fires once every MMA of this CTA has retired
    mbar_wait(b_mmadone, 0);
  }
  __syncwarp();
  fence_before();
  __syncthreads();
  if (warp == 8) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256));
}

}  // namespace

bool tc_attention_supported(int dtype, int D_, int rep) { return dtype == PIC_BF16 && D_ == D && rep == REP; }

void launch_attention_tc(const AttnArgs& a, cudaStream_t st) {
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int smem = SMEM_BYTES + 1024;
  if (dev < 0 || dev >= 64 || !attr[dev]) {
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (dev >= 0 && dev < 64) attr[dev] = true;
  }
  if (a.n_items > 0) attn_tc_kernel<<<a.n_items, kThreads, smem, st>>>(a);
}

pic_status attn_check_timeout() {
  int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_timeout, sizeof(int));
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("timeout flag: ") + cudaGetErrorString(e));
  if (v) {
    cudaMemcpyToSymbol(g_attn_timeout, &zero, sizeof(int));
    return fail(PIC_ERR_DEVICE_TIMEOUT, "the tensor-core attention kernel gave up a bounded wait");
  }
  return PIC_OK;
}

}  // namespace pic
