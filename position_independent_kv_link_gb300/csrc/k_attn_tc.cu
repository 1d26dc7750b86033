// tcgen05 paged attention with fused RoPE for bf16 KV, head_dim 128, 4 query heads per KV head.
//
// Persistent: CTA b walks the work items b, b + grid, b + 2 grid, ... (the planner deals them
// in that order). An item is up to 64 consecutive query rows of one sequence x the 4 query
// heads sharing KV head g x a run of pages. Its rows form two M = 128 MMA tiles: tile t holds
// rows 32t..32t+31 of the item x the 4 heads (MMA row = head * 32 + row). Every 64-key tile
// (4 pages) of K and V is loaded, rotated and converted ONCE and then feeds both MMA tiles,
// which halves the per-row cost of the K rotation against items of 32 rows. Rows are in
// ascending position order, so tile 0 sees no key beyond its own last row: it stops after the
// key tiles holding pages [page0, page_mid) and the item's later key tiles run for tile 1
// alone.
//
//   warp 17     loads: one TMA box per page for its pre-RoPE K and one for its V (16 rows x both
//               64-dim halves, 4 KB, 128-byte swizzled; two key tiles in flight), the cos/sin
//               table rows of the page starts (plain loads by the warp's lanes) and, per item,
//               the Q tiles (rotated and scaled fp16 rows written by the QKV epilogue).
//   warps 8-15  transform: K rotated by RoPE at each key's absolute position (MEPIC abstract:
//               K is kept without positional encoding and RoPE is fused into attention) into
//               the fp16 K-major operand; V converted to fp16 into the MN-major operand of
//               O += P V ([key][dim], three key tiles held until their PV). cos/sin(p theta) is
//               composed from the table row of the page start and that of the offset inside
//               the page (the latter held in registers: each thread always rotates the same
//               row offset and dims).
//   warp 16     TMEM owner (all 512 columns: O of tile t at [128t, 128t + 128), two S buffers
//               of tile t at 256 + 128t + {0, 64}); one thread issues S_t = Q_t K^T (M128 N64
//               K128) and O_t += P_t V (M128 N128 K64, P_t read from TMEM) with tcgen05.mma
//               kind::f16.
//   warps 0-7   softmax: warpgroup t serves MMA tile t, thread = one MMA row = one TMEM lane.
//               Reads its row of S, masks keys after its position (only on key tiles that need
//               it), keeps a running reference maximum and writes P = 2^(S - ref) as fp16
//               pairs over the same S buffer in TMEM, the A operand of the PV product. O in
//               TMEM is rescaled only when the maximum grows by more than 2^8 (P stays <= 256,
//               safe in fp16); the sum uses the same reference, so O / l is exact softmax. At
//               the end of an item it drains O_t (normalized output, or the unnormalized
//               partial with its reference maximum and sum for the merge).
// Barrier phases run over the CTA's whole key-tile sequence (and per MMA tile over that tile's
// own sequence), so the next item's loads overlap the current item's tail. Every wait is
// bounded; on expiry the CTA raises the device timeout flag, stops issuing work, waits
// (bounded) for the TMA copies and MMAs already issued, frees its TMEM and returns.
#include <climits>
#include <mutex>

#include <cudaTypedefs.h>

#include "pic_internal.h"

namespace pic {

bool tc_attention_supported(int dtype, int D, int rep);
void launch_attention_tc(const AttnArgs& a, cudaStream_t st);

namespace {

constexpr int D = 128;
constexpr int REP = 4;
constexpr int RB = 32;                    // query rows per MMA tile
constexpr int MT = 2;                     // MMA tiles per item (items of up to 64 rows)
constexpr int KT = 64;                    // keys per tile (4 pages)
constexpr int NRS = 2;                    // raw K/V tiles in flight (freed once transformed); also
                                          // indexes the page metadata and cos/sin rows of a tile
constexpr int NVS = 3;                    // fp16 V operand tiles (freed once their PVs retired);
                                          // also indexes the key positions of a tile
constexpr int kSoftmaxWarps = 4 * MT;
constexpr int kTransformWarps = 8;
constexpr int W_XF = kSoftmaxWarps;                 // first transform warp
constexpr int W_MMA = W_XF + kTransformWarps, W_LOAD = W_MMA + 1;
constexpr int kThreads = (W_LOAD + 1) * 32;
constexpr float kRescale = 8.f;           // rescale O when the row max grows by more than 2^8
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;

// shared memory map (bytes from a 1024-aligned base)
constexpr int Q_TILE = 32768;                     // one MMA tile of Q: 2 halves x [128 rows][128 B] fp16
constexpr int OFF_Q = 0;                          // [MT] Q tiles                              64 KB
constexpr int OFF_KOP = OFF_Q + MT * Q_TILE;      // [2][2 halves][64 keys][128 B] fp16        32 KB
// raw pages as TMA writes them: [page][16 rows][2 halves][128 B], the 128-byte rows swizzled
constexpr int OFF_KRAW = OFF_KOP + 32768;         // [2][4 pages][4 KB] bf16                   32 KB
constexpr int OFF_VRAW = OFF_KRAW + NRS * 16384;  // [2][4 pages][4 KB] bf16                   32 KB
constexpr int OFF_V = OFF_VRAW + NRS * 16384;     // [3][2 halves][64 keys][128 B] fp16        48 KB
constexpr int OFF_CS = OFF_V + NVS * 16384;       // [2][4 pages][512 B] cos/sin rows           4 KB
constexpr int OFF_TM = OFF_CS + NRS * 2048;       // int [2][4][2] page start, valid rows
constexpr int OFF_POS = OFF_TM + 128;             // int [3][KT] key positions (INT_MAX = none)
constexpr int OFF_TILE = OFF_POS + NVS * KT * 4;  // int [3] last key position, INT_MAX if ragged
constexpr int OFF_BAR = OFF_TILE + 16;
constexpr int N_BARS = 32;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16;
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_BYTES + 1024 <= 227 * 1024, "shared memory budget");

// barrier slots ([t][b]: MMA tile t, S buffer b)
constexpr int B_KVFULL = 0;                       // [2]   K operand buffer ready (transform)
constexpr int B_SFULL = 2;                        // [2][2] S_t in buffer b computed (MMA commit)
constexpr int B_PFULL = 6;                        // [2][2] P_t in buffer b written (softmax t)
constexpr int B_PVDONE = 10;                      // [2][2] O_t += P_t V of buffer b retired (commit)
constexpr int B_RAWFULL = 14;                     // [2]   raw K/V tile landed (TMA)
constexpr int B_RAWFREE = 16;                     // [2]   raw K/V tile consumed (transform)
constexpr int B_VFREE = 18;                       // [3]   V operand slot's PVs retired (commit)
constexpr int B_POSFULL = 21;                     // [3]   key positions of a V slot (transform)
constexpr int B_QFULL = 24, B_QFREE = 25;         // item's Q tiles landed / every S of the item done
constexpr int B_OFREE = 26;                       // [2]   O_t drained (softmax t)
constexpr int B_MMADONE = 28;
constexpr int B_KFREE = 29;                       // [2]   every S of the K operand buffer's tile done (commit)
static_assert(B_KFREE + 2 <= N_BARS, "barrier slots");
// Every waiter must observe each phase of a barrier before the barrier can complete the next
// one (a parity wait cannot tell phase n from n + 2). KVFULL therefore has only the MMA as a
// waiter, and KFREE only the transform (the MMA cannot commit buffer b's next S before the
// transform re-armed KVFULL); the
// softmax takes the key positions from POSFULL, per V slot, which the transform re-arms only
// after every PV of the slot's key tile, i.e. after both softmax warpgroups consumed it. The
// S/P/PV barriers of MMA tile t count that tile's own key tiles, so a warpgroup that skips
// key tiles (tile 0 past page_mid) never waits on phases it did not take part in.

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
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// expected transaction bytes without an arrival (the arrival follows separately)
__device__ __forceinline__ void mbar_add_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// 16-byte chunk c (0..7) of row r of a [rows][128 B] tile, 128-byte swizzle (the TMA and UMMA layout)
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// K-major operand: 8-row atoms 1024 B apart, 128-byte swizzle
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// MN-major operand [k rows][n] (n contiguous, 64 n per 128-byte row): blocks of 64 n are
// `lbo` bytes apart, groups of 8 k rows 1024 B apart, 128-byte swizzle
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16, A and B fp16, D fp32, M x N; A K-major; B K-major or MN-major
__device__ __forceinline__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D (TMEM) [+]= A (shared memory) . B (shared memory)
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// D (TMEM) [+]= A (TMEM: row m in lane m, 16-bit elements 2k and 2k + 1 in column k) . B (shared memory)
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc));
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
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float* v) {
  uint32_t u[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(v[i]);
  tmem_st16(taddr, u);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// bf16 pair -> fp16 pair (exact widening, one rounding)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ void bf8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16);
    f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
  }
}

// key tiles of an item, and those MMA tile t takes part in (tile 0: pages [page0, page_mid);
// tile 1: every key tile when the item has more than 32 rows, none otherwise)
__device__ __forceinline__ int item_tiles(const AttnItem& it) { return (it.page1 - it.page0 + 3) >> 2; }
__device__ __forceinline__ int item_tiles_of(const AttnItem& it, int t) {
  if (t == 0) return max(0, (it.page_mid - it.page0 + 3) >> 2);
  return it.nrows > RB ? item_tiles(it) : 0;
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* sTm = reinterpret_cast<int*>(sm + OFF_TM);   // [slot][page][start, valid rows]
  int* sPos = reinterpret_cast<int*>(sm + OFF_POS);
  int* sTile = reinterpret_cast<int*>(sm + OFF_TILE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + N_BARS);
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_KVFULL + i), kTransformWarps);
      mbar_init(bar(B_KFREE + i), 1);
    }
    for (int i = 0; i < 2 * MT; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PFULL + i), 4);
      mbar_init(bar(B_PVDONE + i), 1);
    }
    for (int i = 0; i < NRS; ++i) {
      mbar_init(bar(B_RAWFULL + i), 1);
      mbar_init(bar(B_RAWFREE + i), kTransformWarps);
    }
    for (int i = 0; i < NVS; ++i) {
      mbar_init(bar(B_VFREE + i), 1);
      mbar_init(bar(B_POSFULL + i), kTransformWarps);
    }
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QFREE), 1);
    for (int t = 0; t < MT; ++t) mbar_init(bar(B_OFREE + t), 4);
    mbar_init(bar(B_MMADONE), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  pdl_enter();   // the setup above overlaps the previous kernel; everything below reads its outputs
  const uint32_t tmem = *tmem_slot;

  if (warp < kSoftmaxWarps) {
    // =============================== softmax warps: warpgroup t, head hh, row r of MMA tile t
    const int t = warp >> 2, hh = warp & 3, r = lane;   // MMA row hh * 32 + r = TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(hh * 32) << 16);   // this warp's TMEM lane quarter
    const uint32_t t_o = trow + 128 * t, t_s = trow + 256 + 128 * t;
    uint32_t gt = 0, ct = 0;   // key tiles of the CTA; key tiles of this MMA tile
    bool ok = true;
    for (int ii = blockIdx.x; ii < a.n_items && ok; ii += gridDim.x) {
      const AttnItem it = a.items[ii];
      const int nt = item_tiles(it), na = item_tiles_of(it, t);
      const int row = RB * t + r;
      if (RB * t >= it.nrows) {   // no rows of this MMA tile in the item (then na == 0)
        gt += nt;
        continue;
      }
      const int qp = row < it.nrows ? a.q_pos[it.row0 + row] : -1;
      float mref = -INFINITY, l = 0.f;
      for (int j = 0; j < na; ++j, ++ct) {
        const uint32_t g = gt + j;
        const int b = ct & 1, sl = g % NVS;
        // S of the key tile, and the transform's key positions of it
        ok = __all_sync(0xffffffffu, !s_abort && mbar_wait(bar(B_SFULL + 2 * t + b), (ct >> 1) & 1) &&
                                         mbar_wait(bar(B_POSFULL + sl), (g / NVS) & 1));
        if (!ok) break;
        fence_after();
        // Two halves of 32 keys keep the register footprint low: the low half is read for the
        // maximum and again for P; P (64 fp16 = 32 columns) goes over the high half's columns,
        // high keys first (their S is in registers by then), then the low keys.
        const uint32_t sb = t_s + 64 * b;
        const bool need_mask = __any_sync(0xffffffffu, sTile[sl] > qp);
        const int* kpos = sPos + sl * KT;
        auto load_half = [&](int h, float* v) {   // S of keys 32h..32h+31, masked by position
          tmem_ld16(sb + 32 * h, v);
          tmem_ld16(sb + 32 * h + 16, v + 16);
          tmem_wait_ld();
          if (need_mask) {
            const int4* kp = reinterpret_cast<const int4*>(kpos + 32 * h);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int4 k4 = kp[i];
              if (k4.x > qp) v[4 * i] = -INFINITY;
              if (k4.y > qp) v[4 * i + 1] = -INFINITY;
              if (k4.z > qp) v[4 * i + 2] = -INFINITY;
              if (k4.w > qp) v[4 * i + 3] = -INFINITY;
            }
          }
        };
        float s[32];
        load_half(0, s);
        float mx = s[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) mx = fmaxf(mx, s[i]);
        load_half(1, s);
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, s[i]);
        // new reference when the maximum grows by more than 2^8 (or for the first keys seen)
        const bool grow = mx > mref + kRescale;
        const float mnew = grow ? mx : mref;
        const float scale = (grow && mref != -INFINITY) ? ex2(mref - mnew) : 1.f;
        l *= scale;
        mref = mnew;
        // P = 2^(S - ref) as fp16 pairs: keys 2c, 2c + 1 in column 32 + c of the S buffer
        const float mz = mref == -INFINITY ? 0.f : mref;   // fully masked so far: every s is -inf, p = 0
        float rs = 0.f;
        auto store_p = [&](int h) {
          uint32_t pv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2(s[2 * e] - mz), p1 = ex2(s[2 * e + 1] - mz);
            rs += p0 + p1;
            pv[e] = pack_f16x2(p0, p1);
          }
          tmem_st16(sb + 32 + 16 * h, pv);
        };
        store_p(1);
        load_half(0, s);
        store_p(0);
        if (__any_sync(0xffffffffu, scale != 1.f)) {
          // O holds the sums of this item's earlier key tiles: rescale it before this P is added,
          // once the PV of the previous key tile has retired (a rescale needs a finite earlier
          // maximum, so j > 0)
          const uint32_t pc = ct - 1;
          if (!mbar_wait(bar(B_PVDONE + 2 * t + (pc & 1)), (pc >> 1) & 1)) ok = false;
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          fence_after();
#pragma unroll 1
          for (int c = 0; c < 128; c += 16) {
            float o[16];
            tmem_ld16(t_o + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= scale;
            tmem_st16f(t_o + c, o);
          }
        }
        l += rs;
        tmem_wait_st();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + 2 * t + b));
      }
      if (!ok) break;
      // ---- drain O_t: normalized output, or the unnormalized partial with its reference max and sum
      if (na > 0) {
        const uint32_t pc = ct - 1;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B_PVDONE + 2 * t + (pc & 1)), (pc >> 1) & 1));
        if (!ok) break;
        fence_after();
      }
      const int h = it.g * REP + hh;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 64) {   // 64 columns per TMEM round trip
        float o[64];
        if (na > 0) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16(t_o + c0 + 16 * c, o + 16 * c);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) o[e] = 0.f;
        }
        if (it.part < 0) {
          if (row < it.nrows) {
            uint4* dst = reinterpret_cast<uint4*>((__half*)a.out + ((size_t)(it.row0 + row) * a.H + h) * D + c0);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[c] = make_uint4(pack_f16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                  pack_f16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                  pack_f16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                  pack_f16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
          }
        } else if (row < it.nrows) {
          float4* dst =
              reinterpret_cast<float4*>(a.part_o + (((size_t)it.part * kAttnPartRows + row) * REP + hh) * D + c0);
#pragma unroll
          for (int e = 0; e < 16; ++e) dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        }
      }
      if (na > 0) {
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_OFREE + t));
      }
      if (it.part >= 0 && row < it.nrows) {
        const size_t pi = ((size_t)it.part * kAttnPartRows + row) * REP + hh;
        *reinterpret_cast<float2*>(a.part_ml + pi * 2) = make_float2(mref, l);
      }
      gt += nt;
    }
    if (!ok) s_abort = 1;
  } else if (warp < W_MMA) {
    // =============================== transform warps
    const int tt = tid - W_XF * 32, tw = warp - W_XF;
    // K: row offset rr of pages pg0, pg0 + 1; dims 8cq..8cq+7 and 64 + 8cq..
    const int rr = lane & 15, cq = 2 * (tw & 3) + (lane >> 4), pg0 = 2 * (tw >> 2);
    float2 lo[8];   // (cos, sin)(rr theta_i) for this thread's 8 frequencies
#pragma unroll
    for (int e = 0; e < 8; ++e) lo[e] = a.rope_cs[rr * 64 + 8 * cq + e];
    uint32_t gt = 0;
    bool ok = true;
    for (int ii = blockIdx.x; ii < a.n_items && ok; ii += gridDim.x) {
      const int nt = item_tiles(a.items[ii]);
      for (int j = 0; j < nt; ++j, ++gt) {
        const int b = gt & 1, rs = gt % NRS, s = gt % NVS;
        const uint32_t u = gt >> 1;
        // raw tile landed; K operand buffer b free once every S of key tile gt - 2 has completed
        // (KVFULL's next phase is taken by the MMA only after those S); V operand slot s (and
        // its key positions) once every PV of key tile gt - 3 has retired
        ok = __all_sync(0xffffffffu, !s_abort && mbar_wait(bar(B_RAWFULL + rs), (gt / NRS) & 1) &&
                                         (gt < 2 || mbar_wait(bar(B_KFREE + b), (u - 1) & 1)) &&
                                         (gt < NVS || mbar_wait(bar(B_VFREE + s), (gt / NVS - 1) & 1)));
        if (!ok) break;
        const int* tm = sTm + rs * 8;
        const uint8_t* kraw = sm + OFF_KRAW + rs * 16384;
        uint8_t* kop = sm + OFF_KOP + b * 16384;
        // K: rotate row offset rr of pages pg0 and pg0 + 1 (two independent chains)
#pragma unroll
        for (int pg = pg0; pg < pg0 + 2; ++pg) {
          const int key = pg * 16 + rr, start = tm[2 * pg], len = tm[2 * pg + 1];
          uint4 y1 = make_uint4(0, 0, 0, 0), y2 = y1;
          if (rr < len) {
            float v1[8], v2[8];
            const uint8_t* kp = kraw + pg * 4096;   // 128-byte rows 2 rr (dims 0..63) and 2 rr + 1
            bf8_to_f32(*reinterpret_cast<const uint4*>(kp + sw128(2 * rr, cq)), v1);
            bf8_to_f32(*reinterpret_cast<const uint4*>(kp + sw128(2 * rr + 1, cq)), v2);
            const float4* hrow = reinterpret_cast<const float4*>(sm + OFF_CS + (rs * 4 + pg) * 512) + 4 * cq;
            uint32_t o1[4], o2[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 h4 = hrow[q];   // (cos, sin) of the page start for frequencies 8cq + 2q, + 1
              const float2 hi[2] = {make_float2(h4.x, h4.y), make_float2(h4.z, h4.w)};
              float y1e[2], y2e[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int f = 2 * q + e;
                const float cs = hi[e].x * lo[f].x - hi[e].y * lo[f].y;
                const float sn = hi[e].y * lo[f].x + hi[e].x * lo[f].y;
                y1e[e] = v1[f] * cs - v2[f] * sn;
                y2e[e] = v2[f] * cs + v1[f] * sn;
              }
              o1[q] = pack_f16x2(y1e[0], y1e[1]);
              o2[q] = pack_f16x2(y2e[0], y2e[1]);
            }
            y1 = make_uint4(o1[0], o1[1], o1[2], o1[3]);
            y2 = make_uint4(o2[0], o2[1], o2[2], o2[3]);
          }
          *reinterpret_cast<uint4*>(kop + sw128(key, cq)) = y1;
          *reinterpret_cast<uint4*>(kop + 8192 + sw128(key, cq)) = y2;
          if (cq == 0) sPos[s * KT + key] = rr < len ? start + rr : INT_MAX;
        }
        if (tt == 0) {   // last key position of the tile; INT_MAX when some slot holds no key
          int kmax = -1;
          bool full = true;
          for (int pg = 0; pg < 4; ++pg) {
            const int len = tm[2 * pg + 1];
            if (len > 0) kmax = tm[2 * pg] + len - 1;
            if (len < kBlock) full = false;
          }
          sTile[s] = full ? kmax : INT_MAX;
        }
        // V: raw [page][row][half] bf16 -> fp16 [half][key][128 B], the MN-major operand; rows
        // without a key become 0 (P is 0 there, V must be finite)
        const uint8_t* vraw = sm + OFF_VRAW + rs * 16384;
        uint8_t* vt = sm + OFF_V + s * 16384;
#pragma unroll
        for (int i = 0; i < 1024 / (32 * kTransformWarps); ++i) {
          const int ch = tt + 32 * kTransformWarps * i;   // 16-byte chunk of the raw tile
          const int pg = ch >> 8, rp = (ch >> 3) & 31, r = rp >> 1, h = rp & 1, c = (ch & 7) ^ (rp & 7);
          const int key = pg * 16 + r;
          uint4 o = make_uint4(0, 0, 0, 0);
          if (r < tm[2 * pg + 1]) {
            const uint4 w = *reinterpret_cast<const uint4*>(vraw + ch * 16);
            o = make_uint4(bf2_to_h2(w.x), bf2_to_h2(w.y), bf2_to_h2(w.z), bf2_to_h2(w.w));
          }
          *reinterpret_cast<uint4*>(vt + h * 8192 + sw128(key, c)) = o;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_RAWFREE + rs));
          mbar_arrive(bar(B_KVFULL + b));
          mbar_arrive(bar(B_POSFULL + s));
        }
      }
    }
    if (!ok) s_abort = 1;
  } else if (warp == W_MMA) {
    // =============================== MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(128, KT, false), id_pv = idesc_f16(128, D, true);
      uint32_t gt = 0, ai = 0;
      uint32_t ct[MT] = {0, 0}, ci[MT] = {0, 0};   // per MMA tile: key tiles and items taken part in
      // S_t of the MMA tile's c-th key tile into S buffer c & 1, from the K operand at kaddr
      auto issue_s = [&](int t, uint32_t c, uint32_t kaddr) -> bool {
        const int b = c & 1;
        // the buffer's previous contents (P of key tile c - 2) must have been read by its PV
        if (c >= 2 && !mbar_wait(bar(B_PVDONE + 2 * t + b), ((c - 2) >> 1) & 1)) return false;
        fence_after();
        const uint32_t qa = smem_u32(sm + OFF_Q + t * Q_TILE);
#pragma unroll
        for (int k = 0; k < 8; ++k) {   // K dimension 128 = 2 halves x 4 steps of 16
          const uint32_t off = (k & 3) * 32;
          umma_ss(tmem + 256 + 128 * t + 64 * b, desc_kmajor(qa + (k >> 2) * 16384 + off),
                  desc_kmajor(kaddr + (k >> 2) * 8192 + off), id_s, k != 0);
        }
        umma_commit(bar(B_SFULL + 2 * t + b));
        return true;
      };
      // every S of key tile g (the item's j-th): its K operand ready, then each MMA tile taking part
      auto issue_tile_s = [&](uint32_t g, int j, const int* na) -> bool {
        const int kb = g & 1;
        if (s_abort || !mbar_wait(bar(B_KVFULL + kb), (g >> 1) & 1)) return false;
        fence_after();
        const uint32_t kaddr = smem_u32(sm + OFF_KOP + kb * 16384);
        for (int t = 0; t < MT; ++t)
          if (j < na[t] && !issue_s(t, ct[t] + j, kaddr)) return false;
        umma_commit(bar(B_KFREE + kb));   // the K operand buffer is free once these S complete
        return true;
      };
      bool ok = true;
      for (int ii = blockIdx.x; ii < a.n_items && ok; ii += gridDim.x) {
        const AttnItem it = a.items[ii];
        const int nt = item_tiles(it);
        const int na[MT] = {item_tiles_of(it, 0), item_tiles_of(it, 1)};
        if (nt == 0) continue;
        if (s_abort || !mbar_wait(bar(B_QFULL), ai & 1)) {
          ok = false;
          break;
        }
        ok = issue_tile_s(gt, 0, na);
        if (ok && nt == 1) umma_commit(bar(B_QFREE));
        for (int j = 0; j < nt && ok; ++j) {
          const uint32_t g = gt + j;
          if (j + 1 < nt) {   // next key tile's S first: the softmax finds it ready after this P
            if (!issue_tile_s(g + 1, j + 1, na)) {
              ok = false;
              break;
            }
            if (j + 2 == nt) umma_commit(bar(B_QFREE));   // every S of this item issued
          }
          const int s = g % NVS;
          const uint32_t vb = smem_u32(sm + OFF_V + s * 16384);
          for (int t = 0; t < MT; ++t) {
            if (j >= na[t]) continue;
            const uint32_t c = ct[t] + j;
            const int b = c & 1;
            if (s_abort || !mbar_wait(bar(B_PFULL + 2 * t + b), (c >> 1) & 1) ||
                (j == 0 && ci[t] > 0 && !mbar_wait(bar(B_OFREE + t), (ci[t] - 1) & 1))) {   // previous O_t drained
              ok = false;
              break;
            }
            fence_after();
            const uint32_t pa = tmem + 256 + 128 * t + 64 * b + 32;   // P over the S buffer's high half
#pragma unroll
            for (int k = 0; k < 4; ++k)   // K dimension 64 keys = 4 steps of 16 (8 TMEM columns of P each)
              umma_ts(tmem + 128 * t, pa + 8 * k, desc_mnmajor(vb + k * 2048, 8192), id_pv, (j | k) != 0);
            umma_commit(bar(B_PVDONE + 2 * t + b));
          }
          if (ok) umma_commit(bar(B_VFREE + s));
        }
        for (int t = 0; t < MT; ++t)
          if (na[t] > 0) {
            ct[t] += na[t];
            ++ci[t];
          }
        gt += nt;
        ++ai;
      }
      if (!ok) s_abort = 1;
      umma_commit(bar(B_MMADONE));   // fires once every MMA of this CTA has retired
      mbar_wait(bar(B_MMADONE), 0);
    }
  } else if (warp == W_LOAD) {
    // =============================== loads (lane 0 issues; the warp reads page metadata)
    uint32_t n_raw = 0, n_q = 0;   // raw key tiles and Q loads issued
    bool ok = true;
    int w0 = 0, wblk = 0, wpos = 0, wlen = 0;   // lane i: metadata of page w0 + i
    for (int ii = blockIdx.x; ii < a.n_items && ok; ii += gridDim.x) {
      const AttnItem it = a.items[ii];
      const int nt = item_tiles(it);
      for (int j = 0; j < nt; ++j) {
        const uint32_t gt = n_raw;
        const int rs = gt % NRS;
        const uint32_t kr = gt / NRS;
        const int p0 = it.page0 + 4 * j, np = min(4, it.page1 - p0);
        if (j == 0 || p0 + 4 > w0 + 32) {
          w0 = p0;
          const int pg = w0 + lane;
          if (pg < it.page1) {
            wblk = a.page_block[pg];
            wpos = a.page_pos[pg];
            wlen = a.page_len[pg];
          }
        }
        int blk[4], pos[4], len[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          blk[q] = __shfl_sync(0xffffffffu, wblk, p0 - w0 + q);
          pos[q] = __shfl_sync(0xffffffffu, wpos, p0 - w0 + q);
          len[q] = q < np ? __shfl_sync(0xffffffffu, wlen, p0 - w0 + q) : 0;
        }
        // raw slot rs free once the transform is done with key tile gt - 2
        if (lane == 0) ok = !s_abort && (kr == 0 || mbar_wait(bar(B_RAWFREE + rs), (kr - 1) & 1));
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // cos/sin rows of the page starts: 4 x 512 B, one 16-byte chunk per lane and page,
        // loaded before the TMA issue so that their latency overlaps it
        float4 cs4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < np) cs4[q] = reinterpret_cast<const float4*>(a.rope_cs + (size_t)pos[q] * 64)[lane];
        const uint32_t fb = bar(B_RAWFULL + rs);
        if (lane == 0) {
          int* tm = sTm + rs * 8;
          for (int q = 0; q < 4; ++q) {
            tm[2 * q] = pos[q];
            tm[2 * q + 1] = len[q];
          }
          mbar_add_tx(fb, (uint32_t)np * 8192);
        }
        __syncwarp();
        if (lane < np) {   // one lane per page issues that page's K and V boxes
          const uint32_t kd = smem_u32(sm + OFF_KRAW + rs * 16384) + lane * 4096,
                         vd = smem_u32(sm + OFF_VRAW + rs * 16384) + lane * 4096;
          const int bq = lane == 0 ? blk[0] : lane == 1 ? blk[1] : lane == 2 ? blk[2] : blk[3];
          const int y = (bq * a.G + it.g) * kBlock;
          tma_3d(kd, &a.kmap, 0, 0, y, fb);
          tma_3d(vd, &a.vmap, 0, 0, y, fb);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < np) reinterpret_cast<float4*>(sm + OFF_CS + (rs * 4 + q) * 512)[lane] = cs4[q];
        __syncwarp();
        if (lane == 0) mbar_arrive(fb);   // releases the metadata and cos/sin rows with the boxes
        ++n_raw;
        if (j == 0) {   // this item's Q tiles, once every S of the previous item has completed
          if (lane == 0) ok = !s_abort && (n_q == 0 || mbar_wait(bar(B_QFREE), (n_q - 1) & 1));
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (lane == 0) {
            const int nq = it.nrows > RB ? 2 : 1;
            const uint32_t qb = bar(B_QFULL);
            mbar_expect_tx(qb, (uint32_t)nq * Q_TILE);
            for (int t = 0; t < nq; ++t)
              for (int q = 0; q < 8; ++q)   // (head, half): 32 rows x 64 dims
                tma_3d(smem_u32(sm + OFF_Q + t * Q_TILE + (q & 1) * 16384 + (q >> 1) * 4096), &a.qmap, 64 * (q & 1),
                       it.g * REP + (q >> 1), it.row0 + RB * t, qb);
          }
          ++n_q;
        }
      }
    }
    if (!ok) s_abort = 1;
    // every copy this CTA issued has landed before its shared memory is given up (on the
    // normal path these waits return at once: the consumers have seen every phase)
    if (lane == 0) {
      for (int rs = 0; rs < NRS; ++rs) {
        const uint32_t n = (n_raw + NRS - 1 - rs) / NRS;
        if (n) mbar_wait(bar(B_RAWFULL + rs), (n - 1) & 1);
      }
      if (n_q) mbar_wait(bar(B_QFULL), (n_q - 1) & 1);
    }
  }
  __syncwarp();
  fence_before();
  __syncthreads();
  if (warp == W_MMA) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

int sm_count() {
  static int n[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 152;
  if (!n[dev] && (cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n[dev] <= 0))
    n[dev] = 152;
  return n[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

bool tc_attention_supported(int dtype, int D_, int rep) { return dtype == PIC_BF16 && D_ == D && rep == REP; }

bool attn_q_map(CUtensorMap* m, const void* q16, int T, int H) {
  auto enc = encode_fn();
  if (!enc || T < 1 || H < 1) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, RB};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(q16), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][128] bf16 viewed as [rows][2 halves][64]: one box = one page (16 rows x both halves)
bool attn_kv_map(CUtensorMap* m, const void* layer, int pool_blocks, int G) {
  auto enc = encode_fn();
  if (!enc || pool_blocks < 1 || G < 1) return false;
  cuuint64_t dims[3] = {64, 2, (cuuint64_t)pool_blocks * G * kBlock};
  cuuint64_t strides[2] = {128, (cuuint64_t)D * 2};
  cuuint32_t box[3] = {64, 2, kBlock};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(layer), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int attention_tc_rows_per_item() { return MT * RB; }

// Grid = min(items, SMs): the planner deals items for exactly this walk.
void launch_attention_tc(const AttnArgs& a, cudaStream_t st) {
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int smem = SMEM_BYTES + 1024;
  if (dev < 0 || dev >= 64 || !attr[dev]) {
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (dev >= 0 && dev < 64) attr[dev] = true;
  }
  if (a.n_items > 0) launch_dependent(attn_tc_kernel, dim3(std::min(a.n_items, sm_count())), dim3(kThreads), smem, st, a);
}

void attn_raise_timeout() {
  const int one = 1;
  cudaMemcpyToSymbol(g_attn_timeout, &one, sizeof(int));
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
