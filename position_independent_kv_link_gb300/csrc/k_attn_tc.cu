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
// Key tiles stream through a ring of 4 shared-memory stages. A stage holds K and V of 64 keys
// exactly in the layout the MMAs read ([64-dim half][key][128 B], 128-byte swizzled): the load
// warp fills each half with one TMA box over 4 consecutive pool blocks (pages of a chunk or a
// query are allocated consecutively), or one box per page when they are not, plus the cos/sin
// table rows of the page starts. The transform then rotates K and converts V to fp16 in place,
// and the stage is free again once the PV products of its key tile have retired.
//
//   warp 17     loads: K and V boxes and the cos/sin rows of each key tile (TMA), the page
//               metadata (the warp's lanes hold a window of 32 pages, the next one prefetched).
//   warps 8-15  transform, in place: K rotated by RoPE at each key's absolute position (MEPIC
//               abstract: K is kept without positional encoding and RoPE is fused into
//               attention) into fp16, V converted to fp16; rows without a key zeroed.
//               cos/sin(p theta) is composed from the table row of the page start and that of
//               the offset inside the page (the latter held in registers: each thread always
//               rotates the same row offset and dims).
//   warp 16     TMEM owner (all 512 columns: O_t at [128t, 128t + 128), two S buffers of tile t
//               at 256 + 128t + {0, 64}); one thread issues the S products S_t = Q_t K^T (M128
//               N64 K128) of both MMA tiles, each as soon as its key tile is transformed and its
//               S buffer free -- a key tile ahead of the softmax.
//   warps 0-7   MMA tile t = warpgroup t, thread = one MMA row = one TMEM lane. The warpgroup
//               writes the tile's Q rows into shared memory at the start of an item (the A
//               operand of its S products); per key tile each thread reads its row of S, masks
//               keys after its position (only on key tiles that need it), keeps a running
//               reference maximum and writes P = 2^(S - ref) as fp16 pairs over the S columns,
//               and the warpgroup's first thread then issues O_t += P_t V (M128 N128 K64, P_t
//               from TMEM) at once. O in TMEM is rescaled only when the maximum grows by more
//               than 2^8 (P stays <= 256, safe in fp16); the sum uses the same reference, so
//               O / l is exact softmax. At the end of an item the warpgroup drains O_t
//               (normalized output, or the unnormalized partial with its reference maximum and
//               sum for the merge).
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
constexpr int NST = 4;                    // key-tile stages
constexpr int kSoftmaxWarps = 4 * MT;
constexpr int kTransformWarps = 8;
constexpr int W_XF = kSoftmaxWarps;                 // first transform warp
constexpr int W_MMA = W_XF + kTransformWarps, W_LOAD = W_MMA + 1;
constexpr int kThreads = (W_LOAD + 1) * 32;
constexpr float kRescale = 8.f;           // rescale O when the row max grows by more than 2^8
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_O = 0, TM_S = 256;  // TMEM columns of O_t (+ 128t) and S buffer b of tile t (+ 128t + 64b)

// shared memory map (bytes from a 1024-aligned base)
constexpr int Q_TILE = 32768;                     // one MMA tile of Q: 2 halves x [128 rows][128 B] fp16
constexpr int ST_BYTES = 32768;                   // one key tile: K then V, each [2 halves][64 keys][128 B]
constexpr int OFF_Q = 0;                          // [MT] Q tiles                              64 KB
constexpr int OFF_ST = OFF_Q + MT * Q_TILE;       // [NST] key-tile stages                    128 KB
constexpr int OFF_CS = OFF_ST + NST * ST_BYTES;   // [NST][4 pages][512 B] cos/sin rows         8 KB
constexpr int OFF_TM = OFF_CS + NST * 2048;       // int [NST][4][2] page start, valid rows
constexpr int OFF_POS = OFF_TM + NST * 32;        // int [NST][KT] key positions (INT_MAX = none)
constexpr int OFF_TILE = OFF_POS + NST * KT * 4;  // int [NST] last key position, INT_MAX if ragged
constexpr int OFF_BAR = (OFF_TILE + NST * 4 + 7) / 8 * 8;
constexpr int N_BARS = 32;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16;
static_assert(SMEM_BYTES + 1024 <= 227 * 1024, "shared memory budget");

// barrier slots ([t][b]: MMA tile t, S buffer b)
constexpr int B_FULL = 0;                         // [NST] stage landed (TMA bytes + loader arrival)
constexpr int B_XF = B_FULL + NST;                // [NST] stage transformed (transform warps)
constexpr int B_EMPTY = B_XF + NST;               // [NST] both MMA tiles' PVs of the stage's key tile retired
constexpr int B_SFULL = B_EMPTY + NST;            // [2][2] S_t in buffer b computed (commit)
constexpr int B_PVDONE = B_SFULL + 2 * MT;        // [2][2] O_t += P_t V of buffer b retired (commit)
constexpr int B_QREADY = B_PVDONE + 2 * MT;       // [2] Q_t of the item written (warpgroup t)
constexpr int B_DONE = B_QREADY + MT;             // [3] every MMA of an issuing thread retired
static_assert(B_DONE + MT + 1 <= N_BARS, "barrier slots");
// Every waiter must observe each phase of a barrier before the barrier can complete the next
// one (a parity wait cannot tell phase n from n + 2). FULL has only the transform as waiter;
// XF is waited on by the S issuer and both warpgroups, but a stage can only be refilled after
// both warpgroups released it, i.e. after each has used that phase (a warpgroup releases a key
// tile it takes no part in only after waiting for it, so its release never counts toward the
// stage's previous use); EMPTY has only the loader. The S/PV/Q barriers of MMA tile t count
// that tile's own key tiles and items: S_t into buffer b is issued only after the PV that read
// buffer b's previous P retired, and the next item's first S_t only after Q_t was rewritten.

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
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
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
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, "
      "%6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
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
  int* sTm = reinterpret_cast<int*>(sm + OFF_TM);   // [stage][page][start, valid rows]
  int* sPos = reinterpret_cast<int*>(sm + OFF_POS);
  int* sTile = reinterpret_cast<int*>(sm + OFF_TILE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + N_BARS);
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(B_FULL + i), 1);
      mbar_init(bar(B_XF + i), kTransformWarps);
      mbar_init(bar(B_EMPTY + i), MT);   // one release per MMA tile
    }
    for (int i = 0; i < 2 * MT; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PVDONE + i), 1);
    }
    for (int t = 0; t < MT; ++t) mbar_init(bar(B_QREADY + t), 1);
    for (int i = 0; i <= MT; ++i) mbar_init(bar(B_DONE + i), 1);
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
  // Programmatic dependent launch: the next kernel may launch now (it waits for this one's
  // completion before reading its outputs). This kernel's own reads of the previous kernels'
  // outputs (the rotated q, the K/V pages) come after griddepcontrol.wait in the roles that make
  // them; the work plan, page tables and cos/sin table are written before the forward starts and
  // are read earlier, overlapping the previous kernel's tail.
  asm volatile("griddepcontrol.launch_dependents;");
  const uint32_t tmem = *tmem_slot;

  if (warp < kSoftmaxWarps) {
    // =============================== MMA tile t: softmax warps (head hh, row r); the warpgroup's
    // first thread issues the tile's PV products
    const int t = warp >> 2, hh = warp & 3, r = lane;   // MMA row hh * 32 + r = TMEM lane
    const bool issuer = hh == 0 && lane == 0;
    const uint32_t trow = tmem + ((uint32_t)(hh * 32) << 16);   // this warp's TMEM lane quarter
    const uint32_t t_o = trow + TM_O + 128 * t, t_sb = trow + TM_S + 128 * t;
    const uint32_t id_pv = idesc_f16(128, D, true);
    uint8_t* qs = sm + OFF_Q + t * Q_TILE;
    // every thread of the warpgroup takes part, so all of them take the same branch after it
    auto wg_all = [&](bool v) -> bool {
      uint32_t res;
      asm volatile(
          "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, %2, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(res)
          : "r"((uint32_t)v), "r"(1 + t)
          : "memory");
      return res != 0;
    };
    uint32_t gt = 0, ct = 0;   // key tiles of the CTA; key tiles of this MMA tile
    bool ok = true;
    const int row = RB * t + r;
    // the next item and this row's position in it are fetched an item ahead
    AttnItem it_n{};
    int qp_n = -1;
    if (blockIdx.x < a.n_items) {
      it_n = a.items[blockIdx.x];
      qp_n = row < it_n.nrows ? a.q_pos[it_n.row0 + row] : -1;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");   // q16 is written by the previous kernel
    for (int ii = blockIdx.x; ii < a.n_items; ii += gridDim.x) {
      const AttnItem it = it_n;
      const int qp = qp_n;
      if (ii + (int)gridDim.x < a.n_items) it_n = a.items[ii + gridDim.x];
      const int nt = item_tiles(it), na = item_tiles_of(it, t);
      const bool mine = row < it.nrows;
      if (na > 0) {
        // this row's q (128 fp16, rotated and scaled) into the K-major, 128-byte-swizzled A
        // operand of the S products: MMA row m = hh * 32 + r, dims 8c..8c+7 of half h at
        // [h][m][chunk c]. Every S product of this tile's previous item has retired (this
        // warpgroup consumed them), and the next is issued only after QREADY.
        const uint4* src =
            reinterpret_cast<const uint4*>(a.q16 + ((size_t)(it.row0 + (mine ? row : 0)) * a.H + it.g * REP + hh) * D);
        const int m = hh * RB + r;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint4 x = mine ? src[c] : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(qs + (c >> 3) * 16384 + sw128(m, c & 7)) = x;
        }
        fence_async_smem();
      }
      ok = wg_all(ok && !s_abort);
      if (!ok) break;
      if (na > 0 && issuer) mbar_arrive(bar(B_QREADY + t));
      float mref = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        const uint32_t g = gt + j;
        const int sl = g % NST;
        if (j >= na) {
          // this MMA tile takes no part in the key tile: release its share of the stage once the
          // stage holds the tile (the release must not count toward the stage's previous use)
          if (issuer) {
            if (!s_abort && mbar_wait(bar(B_XF + sl), (g / NST) & 1))
              umma_commit(bar(B_EMPTY + sl));
            else
              s_abort = 1;
          }
          continue;
        }
        const int b = ct & 1;
        const uint32_t t_s = t_sb + 64 * b;
        bool okw = !s_abort && mbar_wait(bar(B_SFULL + 2 * t + b), (ct >> 1) & 1) &&
                   mbar_wait(bar(B_XF + sl), (g / NST) & 1);
        okw = __all_sync(0xffffffffu, okw);
        if (okw) {
          fence_after();
          // Two halves of 32 keys keep the register footprint low: the low half is read for the
          // maximum and again for P; P (64 fp16 = 32 columns) goes over the high half's columns,
          // high keys first (their S is in registers by then), then the low keys.
          const bool need_mask = __any_sync(0xffffffffu, sTile[sl] > qp);
          const int* kpos = sPos + sl * KT;
          auto load_half = [&](int h, float* v) {   // S of keys 32h..32h+31, masked by position
            tmem_ld16(t_s + 32 * h, v);
            tmem_ld16(t_s + 32 * h + 16, v + 16);
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
            tmem_st16(t_s + 32 + 16 * h, pv);
          };
          store_p(1);
          load_half(0, s);
          store_p(0);
          l += rs;
          if (__any_sync(0xffffffffu, scale != 1.f)) {
            // O holds the sums of this item's earlier key tiles: rescale it before this P is
            // added, once the PV of the previous key tile has retired (a rescale needs a finite
            // earlier maximum, so j > 0)
            if (__all_sync(0xffffffffu, mbar_wait(bar(B_PVDONE + 2 * t + ((ct - 1) & 1)), ((ct - 1) >> 1) & 1))) {
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
            } else {
              okw = false;
            }
          }
          tmem_wait_st();
          fence_before();
        }
        ok = wg_all(okw);   // P_t (and the rescaled O_t) of the whole tile written
        if (!ok) break;
        // ---- O_t += P_t V at once; the stage's share is released when it retires
        if (issuer) {
          fence_after();
          const uint32_t vb = smem_u32(sm + OFF_ST + sl * ST_BYTES + 16384);
          const uint32_t pa = tmem + TM_S + 128 * t + 64 * b + 32;   // P over the S buffer's high half
#pragma unroll
          for (int k = 0; k < 4; ++k)   // K dimension 64 keys = 4 steps of 16 (8 TMEM columns of P each)
            umma_ts(tmem + TM_O + 128 * t, pa + 8 * k, desc_mnmajor(vb + k * 2048, 8192), id_pv, (j | k) != 0);
          umma_commit(bar(B_PVDONE + 2 * t + b));
          umma_commit(bar(B_EMPTY + sl));
        }
        ++ct;
      }
      if (!ok) break;
      if (ii + (int)gridDim.x < a.n_items) qp_n = row < it_n.nrows ? a.q_pos[it_n.row0 + row] : -1;
      // ---- drain O_t: normalized output, or the unnormalized partial with its reference max and sum
      bool okd = true;
      if (na > 0) {
        okd = __all_sync(0xffffffffu, mbar_wait(bar(B_PVDONE + 2 * t + ((ct - 1) & 1)), ((ct - 1) >> 1) & 1));
        fence_after();
      }
      if (okd && RB * t < it.nrows) {
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
            if (mine) {
              uint4* dst = reinterpret_cast<uint4*>((__half*)a.out + ((size_t)(it.row0 + row) * a.H + h) * D + c0);
#pragma unroll
              for (int c = 0; c < 8; ++c)
                dst[c] = make_uint4(pack_f16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                    pack_f16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                    pack_f16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                    pack_f16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
            }
          } else if (mine) {
            float4* dst =
                reinterpret_cast<float4*>(a.part_o + (((size_t)it.part * kAttnPartRows + row) * REP + hh) * D + c0);
#pragma unroll
            for (int e = 0; e < 16; ++e) dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          }
        }
        if (it.part >= 0 && mine) {
          const size_t pi = ((size_t)it.part * kAttnPartRows + row) * REP + hh;
          *reinterpret_cast<float2*>(a.part_ml + pi * 2) = make_float2(mref, l);
        }
        fence_before();   // the next item's first PV overwrites O_t after the barrier at its start
      }
      if (!okd) s_abort = 1;
      gt += nt;
    }
    if (!ok) s_abort = 1;
    // every MMA this thread issued has retired before the TMEM is given up
    if (issuer) {
      umma_commit(bar(B_DONE + t));
      mbar_wait(bar(B_DONE + t), 0);
    }
  } else if (warp == W_MMA) {
    // =============================== S products of both MMA tiles, each as soon as its key tile
    // is transformed, its S buffer free (the PV that read it retired) and, for an item's first,
    // its Q tile written
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(128, KT, false);
      uint32_t gt = 0;
      uint32_t ct[MT] = {0, 0}, ci[MT] = {0, 0};   // per MMA tile: key tiles and items taken part in
      bool ok = true;
      for (int ii = blockIdx.x; ii < a.n_items && ok; ii += gridDim.x) {
        const AttnItem it = a.items[ii];
        const int nt = item_tiles(it);
        const int na[MT] = {item_tiles_of(it, 0), item_tiles_of(it, 1)};
        int js[MT] = {0, 0};
        uint32_t idle = 0;
        unsigned long long t_idle = 0;
        while (js[0] < na[0] || js[1] < na[1]) {
          bool prog = false;
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            if (js[t] >= na[t]) continue;
            const uint32_t g = gt + js[t], c = ct[t] + js[t];
            const int b = c & 1, st = g % NST;
            if (mbar_test(bar(B_XF + st), (g / NST) & 1) &&
                (js[t] > 0 || mbar_test(bar(B_QREADY + t), ci[t] & 1)) &&
                (c < 2 || mbar_test(bar(B_PVDONE + 2 * t + b), ((c - 2) >> 1) & 1))) {
              fence_after();
              const uint32_t qa = smem_u32(sm + OFF_Q + t * Q_TILE), kb = smem_u32(sm + OFF_ST + st * ST_BYTES);
#pragma unroll
              for (int k = 0; k < 8; ++k) {   // K dimension 128 = 2 halves x 4 steps of 16
                const uint32_t off = (k & 3) * 32;
                umma_ss(tmem + TM_S + 128 * t + 64 * b, desc_kmajor(qa + (k >> 2) * 16384 + off),
                        desc_kmajor(kb + (k >> 2) * 8192 + off), id_s, k != 0);
              }
              umma_commit(bar(B_SFULL + 2 * t + b));
              ++js[t];
              prog = true;
            }
          }
          if (prog) {
            idle = 0;
            continue;
          }
          if (idle++ == 0) {
            t_idle = gtimer();
          } else if ((idle & 255) == 0 && (s_abort || gtimer() - t_idle > kWaitLimitNs)) {
            if (!s_abort) atomicExch(&g_attn_timeout, 1);
            ok = false;
            break;
          }
          __nanosleep(64);   // leave the issue slots of this sub-partition to the softmax and transform
        }
        for (int t = 0; t < MT; ++t)
          if (na[t] > 0) {
            ct[t] += na[t];
            ++ci[t];
          }
        gt += nt;
      }
      if (!ok) s_abort = 1;
      umma_commit(bar(B_DONE + MT));   // fires once every MMA of this thread has retired
      mbar_wait(bar(B_DONE + MT), 0);
    }
  } else if (warp < W_MMA) {
    // =============================== transform warps, in place in the stage
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
        const int s = gt % NST;
        ok = __all_sync(0xffffffffu, !s_abort && mbar_wait(bar(B_FULL + s), (gt / NST) & 1));
        if (!ok) break;
        // Every shared-memory input of the tile is read before the first store (the stores go
        // to the same stage, so a load placed after them could not be moved ahead of them).
        const int4 tmA = reinterpret_cast<const int4*>(sTm + s * 8)[0], tmB = reinterpret_cast<const int4*>(sTm + s * 8)[1];
        const int st0 = pg0 ? tmB.x : tmA.x, ln0 = pg0 ? tmB.y : tmA.y, st1 = pg0 ? tmB.z : tmA.z,
                  ln1 = pg0 ? tmB.w : tmA.w;
        uint8_t* kst = sm + OFF_ST + s * ST_BYTES;
        uint8_t* vst = kst + 16384;
        // K, rows rr of pages pg0 and pg0 + 1: dims 8cq..8cq+7 (half 0) and 64 + 8cq.. (half 1)
        uint4* kp[2][2];
        uint4 kr[2][2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int key = (pg0 + u) * 16 + rr;
          kp[u][0] = reinterpret_cast<uint4*>(kst + sw128(key, cq));
          kp[u][1] = reinterpret_cast<uint4*>(kst + 8192 + sw128(key, cq));
          kr[u][0] = *kp[u][0];
          kr[u][1] = *kp[u][1];
        }
        // V: 4 chunks of 16 bytes of [half][key][8]
        uint4 vr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) vr[i] = reinterpret_cast<const uint4*>(vst)[tt + 32 * kTransformWarps * i];
        // K rotated by RoPE at start + rr; rows without a key (ragged or missing pages) become 0
        uint4 ky[2][2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int len = u ? ln1 : ln0;
          ky[u][0] = ky[u][1] = make_uint4(0, 0, 0, 0);
          if (rr < len) {
            float v1[8], v2[8];
            bf8_to_f32(kr[u][0], v1);
            bf8_to_f32(kr[u][1], v2);
            const float4* hrow = reinterpret_cast<const float4*>(sm + OFF_CS + (s * 4 + pg0 + u) * 512) + 4 * cq;
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
            ky[u][0] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
            ky[u][1] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
          }
        }
        // V bf16 -> fp16 in place ([half][key][128 B] is already the MN-major operand of
        // O += P V); rows without a key become 0 (P is 0 there, V must be finite)
        uint4 vy[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = ((tt + 32 * kTransformWarps * i) >> 3) & 63;
          const uint4 w = vr[i];
          const int pg = key >> 4, ln = pg == 0 ? tmA.y : pg == 1 ? tmA.w : pg == 2 ? tmB.y : tmB.w;
          vy[i] = (key & 15) < ln
                      ? make_uint4(bf2_to_h2(w.x), bf2_to_h2(w.y), bf2_to_h2(w.z), bf2_to_h2(w.w))
                      : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          *kp[u][0] = ky[u][0];
          *kp[u][1] = ky[u][1];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(vst)[tt + 32 * kTransformWarps * i] = vy[i];
        if (cq == 0) {
          sPos[s * KT + pg0 * 16 + rr] = rr < ln0 ? st0 + rr : INT_MAX;
          sPos[s * KT + (pg0 + 1) * 16 + rr] = rr < ln1 ? st1 + rr : INT_MAX;
        }
        if (tt == 0) {   // last key position of the tile; INT_MAX when some slot holds no key
          const int sts[4] = {tmA.x, tmA.z, tmB.x, tmB.z}, lns[4] = {tmA.y, tmA.w, tmB.y, tmB.w};
          int kmax = -1;
          bool full = true;
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) {
            if (lns[pg] > 0) kmax = sts[pg] + lns[pg] - 1;
            if (lns[pg] < kBlock) full = false;
          }
          sTile[s] = full ? kmax : INT_MAX;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_XF + s));
      }
    }
    if (!ok) s_abort = 1;
  } else if (warp == W_LOAD) {
    // =============================== loads (lanes issue the boxes; the warp holds page metadata)
    uint32_t n_ld = 0;   // key tiles issued
    bool ok = true;
    // lane i: metadata of page w0 + i (cur) and of page w0 + 32 + i (nxt, loaded one window ahead)
    int w0 = 0, cblk = 0, cpos = 0, clen = 0, nblk = 0, npos = 0, nlen = 0;
    for (int ii = blockIdx.x; ii < a.n_items && ok; ii += gridDim.x) {
      const AttnItem it = a.items[ii];
      const int nt = item_tiles(it);
      auto fetch = [&](int w, int& b, int& p, int& l) {
        const int pg = w + lane;
        if (pg < it.page1) {
          b = a.page_block[pg];
          p = a.page_pos[pg];
          l = a.page_len[pg];
        }
      };
      for (int j = 0; j < nt; ++j) {
        const uint32_t gt = n_ld;
        const int s = gt % NST;
        const uint32_t kr = gt / NST;
        const int p0 = it.page0 + 4 * j, np = min(4, it.page1 - p0);
        if (j == 0) {
          w0 = p0;
          fetch(w0, cblk, cpos, clen);
          fetch(w0 + 32, nblk, npos, nlen);
        } else if (p0 == w0 + 32) {   // windows are 8 key tiles: a tile never straddles two
          w0 = p0;
          cblk = nblk, cpos = npos, clen = nlen;
          fetch(w0 + 32, nblk, npos, nlen);
        }
        int blk[4], pos[4], len[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          blk[q] = __shfl_sync(0xffffffffu, cblk, p0 - w0 + q);
          pos[q] = __shfl_sync(0xffffffffu, cpos, p0 - w0 + q);
          len[q] = q < np ? __shfl_sync(0xffffffffu, clen, p0 - w0 + q) : 0;
        }
        if (gt == 0) asm volatile("griddepcontrol.wait;" ::: "memory");   // the pages are written by earlier kernels
        // stage s free once every PV of key tile gt - NST has retired
        if (lane == 0) ok = !s_abort && (kr == 0 || mbar_wait(bar(B_EMPTY + s), (kr - 1) & 1));
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t fb = bar(B_FULL + s);
        if (lane == 0) {
          int* tm = sTm + s * 8;
          for (int q = 0; q < 4; ++q) {
            tm[2 * q] = pos[q];
            tm[2 * q + 1] = len[q];
          }
          mbar_expect_tx(fb, (uint32_t)np * (8192 + 512));   // arrives too: the boxes complete the phase
        }
        __syncwarp();
        const uint32_t kd = smem_u32(sm + OFF_ST + s * ST_BYTES), vd = kd + 16384;
        const uint32_t csd = smem_u32(sm + OFF_CS + s * 2048);
        const bool run = np == 4 && blk[1] == blk[0] + 1 && blk[2] == blk[0] + 2 && blk[3] == blk[0] + 3;
        if (run) {   // 4 consecutive blocks: one box per (K or V, half), 8 KB each
          if (lane < 4) {
            const int h = lane & 1;
            tma_5d((lane < 2 ? kd : vd) + h * 8192, lane < 2 ? &a.kmap : &a.vmap, 0, h, 0, it.g, blk[0], fb);
          }
        } else if (lane < 4 * np) {   // one box per (page, K or V, half), 2 KB each
          const int q = lane >> 2, h = lane & 1, isv = (lane >> 1) & 1;
          const int bq = q == 0 ? blk[0] : q == 1 ? blk[1] : q == 2 ? blk[2] : blk[3];
          tma_5d((isv ? vd : kd) + h * 8192 + q * 2048, isv ? &a.vmap1 : &a.kmap1, 0, h, 0, it.g, bq, fb);
        }
        if (lane >= 16 && lane < 16 + np) {   // cos/sin rows of the page starts, 512 B each
          const int q = lane - 16;
          const int pq = q == 0 ? pos[0] : q == 1 ? pos[1] : q == 2 ? pos[2] : pos[3];
          tma_2d(csd + q * 512, &a.csmap, 0, pq, fb);
        }
        ++n_ld;
      }
    }
    if (!ok) s_abort = 1;
    // every copy this CTA issued has landed before its shared memory is given up (on the
    // normal path these waits return at once: the consumers have seen every phase)
    if (lane == 0)
      for (int s = 0; s < NST; ++s) {
        const uint32_t n = (n_ld + NST - 1 - s) / NST;
        if (n) mbar_wait(bar(B_FULL + s), (n - 1) & 1);
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

// One layer of a pool, [blocks][G][16 rows][128] bf16, viewed as (64 dims, 2 halves, 16 rows, G,
// blocks): a box is one 64-dim half of the 16 rows of one KV head's page in 4 consecutive blocks
// (m4) or in one block (m1), landing as [pages][16 rows][128 B] -- one half of the K-major (K)
// or MN-major (V) operand of 64 keys.
bool attn_kv_map(CUtensorMap* m4, CUtensorMap* m1, const void* layer, int pool_blocks, int G) {
  auto enc = encode_fn();
  if (!enc || pool_blocks < 1 || G < 1) return false;
  cuuint64_t dims[5] = {64, 2, (cuuint64_t)kBlock, (cuuint64_t)G, (cuuint64_t)pool_blocks};
  cuuint64_t strides[4] = {128, (cuuint64_t)D * 2, (cuuint64_t)kBlock * D * 2, (cuuint64_t)G * kBlock * D * 2};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  cuuint32_t box4[5] = {64, 1, kBlock, 1, 4}, box1[5] = {64, 1, kBlock, 1, 1};
  auto make = [&](CUtensorMap* m, cuuint32_t* box) {
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(layer), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  return make(m4, box4) && make(m1, box1);
}

bool attn_cs_map(CUtensorMap* m, const float2* rope_cs, int n_pos) {
  auto enc = encode_fn();
  if (!enc || n_pos < 1) return false;
  cuuint64_t dims[2] = {D, (cuuint64_t)n_pos};   // D floats = D/2 (cos, sin) pairs per position
  cuuint64_t strides[1] = {(cuuint64_t)D * 4};
  cuuint32_t box[2] = {D, 1}, estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float2*>(rope_cs), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
