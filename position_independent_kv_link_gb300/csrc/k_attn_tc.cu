// tcgen05 paged attention with fused RoPE for bf16 KV, head_dim 128, 4 query heads per KV head.
//
// One cooperative launch per layer, two phases. Phase 1: the CTAs rotate the K of every page of
// the work by RoPE at each row's absolute position (MEPIC abstract: K is kept without positional
// encoding and rotated inside attention) into an fp16 scratch [pages][G][16][128] indexed by the
// work's page number, rows beyond a page's length zero: each page is rotated once per layer
// however many work items read it. A grid barrier follows. Phase 2 reads the rotated K and the
// stored bf16 V straight into the MMA operand layouts by TMA; nothing is converted on the way.
//
// Phase 2 is persistent: CTA b walks the work items b, b + grid, b + 2 grid, ... (the
// planner deals them in that order). An item is up to 64 consecutive query rows of one sequence
// x the 4 query heads sharing KV head g x a run of pages. Its rows form two M = 128 MMA tiles:
// tile t holds rows 32t..32t+31 of the item x the 4 heads (MMA row = head * 32 + row). Every
// 64-key tile (4 pages) of K and V feeds both MMA tiles. Rows are in ascending position order,
// so tile 0 sees no key beyond its own last row: it stops after the key tiles holding pages
// [page0, page_mid) and the item's later key tiles run for tile 1 alone.
//
// Key tiles stream through a ring of 4 shared-memory stages, each K then V of 64 keys in the
// layout the MMAs read ([64-dim half][key][128 B], 128-byte swizzled).
//
//   warp 10     loads: it alone waits at the grid barrier (the other roles read nothing of
//               what other CTAs wrote in phase 1), then per key tile, rotated K as two boxes of 4 consecutive scratch pages (one per
//               64-dim half) and V as two boxes over 4 consecutive pool blocks (pages of a chunk
//               or a query are allocated consecutively), else one box per full page; a page with
//               fewer than 16 rows is copied by the warp's lanes with its missing rows zeroed,
//               and the V rows of pages past the item's end are zeroed (P is 0 there; V must be
//               finite). The warp also writes each key's position (the causal mask) and holds the
//               page metadata (its lanes hold a window of 32 pages, the next one prefetched; the
//               first item's is fetched before phase 1).
//   warps 8, 9  one MMA-issuing thread per MMA tile t (warp 8 also owns the TMEM: all 512
//               columns, O_t at [128t, 128t + 128), two S buffers of tile t at 256 + 128t +
//               {0, 64}). Per key tile j of its tile, in this order: O_t += P_t(j) V(j) (M128 N128
//               K64, bf16, P_t from TMEM) as soon as the warpgroup has written P_t(j), then
//               S_t(j + 2) = Q_t K(j + 2)^T (M128 N64 K128, fp16) into the S buffer that held
//               P_t(j) as soon as key tile j + 2 has landed. One thread's MMAs run in issue order,
//               so that S product cannot overwrite P_t(j) before the PV has read it: no wait for
//               the PV to retire, and the S products stay two key tiles ahead of the softmax.
//   warps 0-7   MMA tile t = warpgroup t, thread = one MMA row = one TMEM lane. The warpgroup
//               writes the tile's Q rows into shared memory at the start of an item (the A
//               operand of its S products; the first item's while the grid barrier is pending); per key tile each thread reads its row of S (64
//               keys, one TMEM round trip), masks keys after its position (only on key tiles
//               that need it), keeps a running reference maximum and writes P = 2^(S - ref) as
//               bf16 pairs over the S columns. O in TMEM is rescaled only when the maximum grows
//               by more than 2^8 (P stays <= 256); the sum uses the same reference, so O / l is
//               exact softmax. At the end of an item each warp drains its rows of O_t (normalized
//               output, or for a split item O / l in fp16 with its reference maximum and sum
//               for the merge).
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
constexpr int W_MMA = kSoftmaxWarps, W_LOAD = W_MMA + MT;   // one MMA-issuing warp per MMA tile
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
constexpr int OFF_POS = OFF_ST + NST * ST_BYTES;  // int [NST][KT] key positions (INT_MAX = none)
constexpr int OFF_TILE = OFF_POS + NST * KT * 4;  // int [NST] last key position, INT_MAX if ragged
constexpr int OFF_BAR = (OFF_TILE + NST * 4 + 7) / 8 * 8;
constexpr int N_BARS = 32;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16;
static_assert(SMEM_BYTES + 1024 <= 227 * 1024, "shared memory budget");

// barrier slots ([t][b]: MMA tile t, S buffer b)
constexpr int B_FULL = 0;                         // [NST] stage landed (TMA bytes + loader arrival)
constexpr int B_EMPTY = B_FULL + NST;             // [NST] both MMA tiles' PVs of the stage's key tile retired
constexpr int B_SFULL = B_EMPTY + NST;            // [2][2] S_t in buffer b computed (commit)
constexpr int B_PVDONE = B_SFULL + 2 * MT;        // [2][2] O_t += P_t V of buffer b retired (commit)
constexpr int B_QREADY = B_PVDONE + 2 * MT;       // [2] Q_t of the item written (the 4 warps of warpgroup t)
constexpr int B_PREADY = B_QREADY + MT;           // [2][2] P_t in buffer b written (the 4 warps of warpgroup t)
constexpr int B_DONE = B_PREADY + 2 * MT;         // [2] every MMA of MMA tile t's issuing thread retired
constexpr int B_ROT = B_DONE + MT;                // [2] a batch of phase 1 (K pages, cos/sin rows) landed in buffer i
static_assert(B_ROT + 2 <= N_BARS, "barrier slots");
// Every waiter must observe each phase of a barrier before the barrier can complete the next
// one (a parity wait cannot tell phase n from n + 2). FULL is waited on by both MMA threads and
// both warpgroups, but a stage can only be refilled after both MMA tiles released it (the PV
// retired, or the key tile was waited for and skipped), i.e. after each has used that phase.
// EMPTY has only the loader. SFULL_t(b) is waited on by the four warps of warpgroup t; the next
// S product into buffer b follows the PV of P_t in b, which waits for all four warps' PREADY, so
// every warp has seen the phase. PREADY_t(b) is waited on by MMA thread t only, and a warp
// writes the next P into b only after that S product. PVDONE is waited on by the warpgroup
// (rescale, drain) and completes once per PV, each after this warpgroup's P. QREADY_t is waited
// on by MMA thread t before an item's first S product, and completes once per item.

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
// plain bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
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
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// kind::f16 with A and B bf16, D fp32, M x N; A K-major (TMEM); B MN-major
__device__ __forceinline__ constexpr uint32_t idesc_bf16_bmn(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// key tiles of an item, and those MMA tile t takes part in (tile 0: pages [page0, page_mid);
// tile 1: every key tile when the item has more than 32 rows, none otherwise)
__device__ __forceinline__ int item_tiles(const AttnItem& it) { return (it.page1 - it.page0 + 3) >> 2; }
__device__ __forceinline__ int item_tiles_of(const AttnItem& it, int t) {
  if (t == 0) return max(0, (it.page_mid - it.page0 + 3) >> 2);
  return it.nrows > RB ? item_tiles(it) : 0;
}

// page metadata of page pg of an item ending at page1 (left as they are past the end)
__device__ __forceinline__ void fetch_page(const AttnArgs& a, int page1, int pg, int& b, int& p, int& l) {
  if (pg < page1) {
    b = a.page_block[pg];
    p = a.page_pos[pg];
    l = a.page_len[pg];
  }
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
      mbar_init(bar(B_EMPTY + i), MT);   // one release per MMA tile
    }
    for (int i = 0; i < 2 * MT; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PVDONE + i), 1);
    }
    for (int t = 0; t < MT; ++t) mbar_init(bar(B_QREADY + t), 4);
    for (int i = 0; i < 2 * MT; ++i) mbar_init(bar(B_PREADY + i), 4);
    for (int t = 0; t < MT; ++t) mbar_init(bar(B_DONE + t), 1);
    mbar_init(bar(B_ROT), 1);
    mbar_init(bar(B_ROT + 1), 1);
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
  // Programmatic dependent launch: the next kernel may launch once every CTA of this one has
  // executed launch_dependents, i.e. once every CTA of this grid is resident (so the next
  // kernel's CTAs can never hold an SM a CTA of this grid still needs for the grid barrier
  // below); this kernel waits for the previous kernels (the K/V pages, the rotated q) before its
  // first read of their outputs.
  asm volatile("griddepcontrol.launch_dependents;");
  const uint32_t tmem = *tmem_slot;
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // The first item of each role and its page metadata are fetched now, so that their load
  // latency passes during phase 1. Softmax warps: MMA tile t, head hh, row r of the item.
  const int t = warp >> 2, hh = warp & 3, r = lane;
  const int row = RB * t + r;
  AttnItem it_n{};   // softmax warps: the next item; load warp: the first item
  int qp_n = -1;
  int cblk = 0, cpos = 0, clen = 0, nblk = 0, npos = 0, nlen = 0;   // load warp: lane i holds pages w0 + i, w0 + 32 + i
  if (blockIdx.x < a.n_items) {
    if (warp < kSoftmaxWarps) {
      it_n = a.items[blockIdx.x];
      qp_n = row < it_n.nrows ? a.q_pos[it_n.row0 + row] : -1;
    } else if (warp == W_LOAD) {
      it_n = a.items[blockIdx.x];
      fetch_page(a, it_n.page1, it_n.page0 + lane, cblk, cpos, clen);
      fetch_page(a, it_n.page1, it_n.page0 + 32 + lane, nblk, npos, nlen);
    }
  }

  // =============================== phase 1: RoPE. The CTAs rotate the K of every page of the work
  // to each row's absolute position (MEPIC abstract: K is kept without positional encoding and
  // rotated inside attention), each a share of the (page, KV head, row, 8-dim chunk) units, into
  // the fp16 scratch krot[page][g][16][128] (rows beyond a page's length zero), so that a page is
  // rotated once however many work items read it; then all CTAs meet at a grid barrier (the
  // launch is cooperative: every CTA is resident), after which phase 2 reads the scratch by TMA.
  {
    // CTA b takes the (page, KV head) pairs [P b / grid, P (b + 1) / grid), page-major, in batches
    // of up to 16 through two buffers (each: two key-tile stages for the pairs' K pages, 4 KB each,
    // and one Q tile for the pages' cos/sin rows, 512 B per row; all idle until phase 2). The next
    // batch's bulk copies are in flight while every thread rotates (row, 8-dim chunk) units of
    // the current one from shared memory into the scratch.
    constexpr int kRotPairs = 2 * ST_BYTES / 4096;   // 16 per buffer
    constexpr int kRotPages = Q_TILE / 8192;         // 4 pages of cos/sin rows per buffer
    const __nv_bfloat16* kl = static_cast<const __nv_bfloat16*>(a.k_layer);
    const int P = a.n_pages * a.G;
    const int pa = (int)((long long)P * blockIdx.x / gridDim.x), pb = (int)((long long)P * (blockIdx.x + 1) / gridDim.x);
    // batch extent from b0: at most kRotPairs pairs over at most kRotPages pages
    auto batch_n = [&](int b0) { return min(min(kRotPairs, pb - b0), (b0 / a.G + kRotPages) * a.G - b0); };
    auto issue = [&](int b0, int buf) {   // warp 0: the batch's copies into buffer buf
      const int n = batch_n(b0), p_lo = b0 / a.G, p_hi = (b0 + n - 1) / a.G;
      uint8_t* ks = sm + OFF_ST + buf * 2 * ST_BYTES;
      uint8_t* css = sm + OFF_Q + buf * Q_TILE;
      uint32_t bytes = (uint32_t)n * 4096u;
      for (int p = p_lo; p <= p_hi; ++p) bytes += (uint32_t)a.page_len[p] * 512u;
      if (lane == 0) mbar_expect_tx(bar(B_ROT + buf), bytes);
      __syncwarp();
      for (int i = lane; i < n; i += 32) {   // K of pair b0 + i: [16 rows][128] bf16 = 4 KB
        const int pg = b0 + i, p = pg / a.G, g = pg % a.G;
        bulk_g2s(smem_u32(ks + i * 4096), kl + ((size_t)a.page_block[p] * a.G + g) * kBlock * D, 4096u, bar(B_ROT + buf));
      }
      for (int p = p_lo + lane; p <= p_hi; p += 32)   // cos/sin rows of the page's valid rows
        bulk_g2s(smem_u32(css + (p - p_lo) * 8192), a.rope_cs + (size_t)a.page_pos[p] * (D / 2),
                 (uint32_t)a.page_len[p] * 512u, bar(B_ROT + buf));
    };
    if (warp == 0 && pa < pb) issue(pa, 0);
    uint32_t ph[2] = {0, 0};
    for (int b0 = pa, k = 0; b0 < pb; b0 += batch_n(b0), ++k) {
      const int buf = k & 1, n = batch_n(b0), nb = b0 + n;
      // the other buffer was last read in the previous batch, which every thread has finished
      if (warp == 0 && nb < pb) issue(nb, buf ^ 1);
      const bool landed = __syncthreads_and(mbar_wait(bar(B_ROT + buf), ph[buf]));   // the same decision in every thread
      ph[buf] ^= 1;
      if (!landed) {
        s_abort = 1;
        break;
      }
      const int p_lo = b0 / a.G;
      const uint8_t* ks = sm + OFF_ST + buf * 2 * ST_BYTES;
      const uint8_t* css = sm + OFF_Q + buf * Q_TILE;
      for (int u = tid; u < n * kBlock * 8; u += kThreads) {
        const int c = u & 7, r = (u >> 3) & (kBlock - 1), i = u >> 7;
        const int pg = b0 + i, p = pg / a.G;
        uint4 y1 = make_uint4(0, 0, 0, 0), y2 = y1;
        if (r < a.page_len[p]) {
          const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(ks + i * 4096) + r * D + 8 * c;
          const uint4 u1 = *reinterpret_cast<const uint4*>(src), u2 = *reinterpret_cast<const uint4*>(src + 64);
          const float4* f4 = reinterpret_cast<const float4*>(css + (p - p_lo) * 8192 + r * 512) + 4 * c;
          const uint32_t w1[4] = {u1.x, u1.y, u1.z, u1.w}, w2[4] = {u2.x, u2.y, u2.z, u2.w};
          uint32_t o1[4], o2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 f = f4[e];   // (cos, sin) of frequencies 8c + 2e and 8c + 2e + 1
            // bf16 pair -> two floats (exact), then the rotate-half pairs (i, i + 64)
            const float a0 = __uint_as_float(w1[e] << 16), a1 = __uint_as_float(w1[e] & 0xffff0000u);
            const float b0v = __uint_as_float(w2[e] << 16), b1 = __uint_as_float(w2[e] & 0xffff0000u);
            o1[e] = pack_f16x2(a0 * f.x - b0v * f.y, a1 * f.z - b1 * f.w);
            o2[e] = pack_f16x2(b0v * f.x + a0 * f.y, b1 * f.z + a1 * f.w);
          }
          y1 = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          y2 = make_uint4(o2[0], o2[1], o2[2], o2[3]);
        }
        __half* dst = a.krot + ((size_t)pg * kBlock + r) * D + 8 * c;   // [page][g] pairs are consecutive
        *reinterpret_cast<uint4*>(dst) = y1;
        *reinterpret_cast<uint4*>(dst + 64) = y2;
      }
      fence_async_smem();   // these generic reads come before the async-proxy copies that reuse the buffer
      __syncthreads();      // this buffer is read before the batch after next is copied into it
    }
    if (s_abort && warp == 0 && lane == 0)   // copies still in flight land before the memory is reused
      for (int q = 0; q < 2; ++q) mbar_wait(bar(B_ROT + q), ph[q]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // phase 2's TMA loads rewrite these stages
    asm volatile("fence.proxy.async.global;" ::: "memory");   // the TMA loads of phase 2 read these rows
    __threadfence();
    __syncthreads();
  }
  // From here the roles run on their own. Only the load warp reads what other CTAs wrote in
  // phase 1, so only it waits at the grid barrier; the first item's Q is written meanwhile.

  if (warp < kSoftmaxWarps) {
    // =============================== MMA tile t: softmax warps (head hh, row r); the warpgroup's
    // first thread issues the tile's PV products
    const bool issuer = hh == 0 && lane == 0;
    const uint32_t trow = tmem + ((uint32_t)(hh * 32) << 16);   // this warp's TMEM lane quarter
    const uint32_t t_o = trow + TM_O + 128 * t, t_sb = trow + TM_S + 128 * t;
    uint8_t* qs = sm + OFF_Q + t * Q_TILE;
    // every thread of the warpgroup takes part, so all of them take the same branch after it
    uint32_t gt = 0, ct = 0;   // key tiles of the CTA; key tiles of this MMA tile
    bool ok = true;
    // the next item and this row's position in it are fetched an item ahead
    // this row's q of item itq (128 fp16, rotated and scaled) into the K-major, 128-byte-swizzled
    // A operand of the S products: MMA row m = hh * 32 + r, dims 8c..8c+7 of half h at
    // [h][m][chunk c]; every load is issued before the first store. Called once every S product
    // of this tile's previous item has retired (this warp consumed the last one), so the next
    // item's Q is in place while the current item's last PV and drain run; its S products are
    // issued only after QREADY.
    auto write_q = [&](const AttnItem& itq) {
      if (item_tiles_of(itq, t) <= 0) return;
      const bool mq = row < itq.nrows;
      const uint4* src =
          reinterpret_cast<const uint4*>(a.q16 + ((size_t)(itq.row0 + (mq ? row : 0)) * a.H + itq.g * REP + hh) * D);
      uint4 x[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) x[c] = mq ? src[c] : make_uint4(0, 0, 0, 0);
      const int m = hh * RB + r;
#pragma unroll
      for (int c = 0; c < 16; ++c) *reinterpret_cast<uint4*>(qs + (c >> 3) * 16384 + sw128(m, c & 7)) = x[c];
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QREADY + t));
    };
    if (blockIdx.x < a.n_items && !s_abort) write_q(it_n);
    for (int ii = blockIdx.x; ii < a.n_items; ii += gridDim.x) {
      const AttnItem it = it_n;
      const int qp = qp_n;
      const bool has_next = ii + (int)gridDim.x < a.n_items;
      if (has_next) it_n = a.items[ii + gridDim.x];
      const int nt = item_tiles(it), na = item_tiles_of(it, t);
      const bool mine = row < it.nrows;
      if (s_abort) {
        ok = false;
        break;
      }
      float mref = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        const uint32_t g = gt + j;
        const int sl = g % NST;
        if (j >= na) {
          // this MMA tile takes no part in the key tile: release its share of the stage once the
          // stage holds the tile (the release must not count toward the stage's previous use)
          if (issuer) {
            if (!s_abort && mbar_wait(bar(B_FULL + sl), (g / NST) & 1))
              umma_commit(bar(B_EMPTY + sl));
            else
              s_abort = 1;
          }
          continue;
        }
        const int b = ct & 1;
        const uint32_t t_s = t_sb + 64 * b;
        bool okw = !s_abort && mbar_wait(bar(B_SFULL + 2 * t + b), (ct >> 1) & 1) &&
                   mbar_wait(bar(B_FULL + sl), (g / NST) & 1);
        okw = __all_sync(0xffffffffu, okw);
        if (!okw) {
          ok = false;
          break;
        }
        {
          fence_after();
          // All 64 keys of the row in registers (one TMEM round trip); P (64 bf16 = 32 columns)
          // goes over the S buffer's high half.
          const bool need_mask = __any_sync(0xffffffffu, sTile[sl] > qp);
          float s[KT];
#pragma unroll
          for (int c = 0; c < KT; c += 16) tmem_ld16(t_s + c, s + c);
          tmem_wait_ld();
          if (need_mask) {
            const int4* kp = reinterpret_cast<const int4*>(sPos + sl * KT);
#pragma unroll
            for (int i = 0; i < KT / 4; ++i) {
              const int4 k4 = kp[i];
              if (k4.x > qp) s[4 * i] = -INFINITY;
              if (k4.y > qp) s[4 * i + 1] = -INFINITY;
              if (k4.z > qp) s[4 * i + 2] = -INFINITY;
              if (k4.w > qp) s[4 * i + 3] = -INFINITY;
            }
          }
          // maximum and sum as 8 independent chains (no long dependent latency chain)
          float m8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) m8[u] = s[u];
#pragma unroll
          for (int i = 8; i < KT; ++i) m8[i & 7] = fmaxf(m8[i & 7], s[i]);
          const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
          // new reference when the maximum grows by more than 2^8 (or for the first keys seen)
          const bool grow = mx > mref + kRescale;
          const float mnew = grow ? mx : mref;
          const float scale = (grow && mref != -INFINITY) ? ex2(mref - mnew) : 1.f;
          l *= scale;
          mref = mnew;
          // P = 2^(S - ref) as bf16 pairs: keys 2c, 2c + 1 in column 32 + c of the S buffer
          const float mz = mref == -INFINITY ? 0.f : mref;   // fully masked so far: every s is -inf, p = 0
          float r8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p0 = ex2(s[32 * h + 2 * e] - mz), p1 = ex2(s[32 * h + 2 * e + 1] - mz);
              r8[e & 7] += p0 + p1;
              pv[e] = pack_bf16x2(p0, p1);
            }
            tmem_st16(t_s + 32 + 16 * h, pv);
          }
          const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
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
              ok = false;
            }
          }
          tmem_wait_st();
          fence_before();
        }
        if (!ok) break;
        // this warp's rows of P_t (and of the rescaled O_t) are written: the MMA thread issues
        // O_t += P_t V once all four warps of the warpgroup have arrived
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PREADY + 2 * t + b));
        ++ct;
      }
      if (!ok) break;
      if (has_next) {
        write_q(it_n);   // every S product of this item has been consumed by this warp
        qp_n = row < it_n.nrows ? a.q_pos[it_n.row0 + row] : -1;
      }
      // ---- drain O_t: normalized output, or (split item) O / l in fp16 with its reference max and sum
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
          } else if (mine) {   // split partial: O / l in fp16 (within V's range), merged with (max, l)
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(a.part_o) +
                                                  (((size_t)it.part * kAttnPartRows + row) * REP + hh) * D + c0);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[c] = make_uint4(pack_f16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                  pack_f16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                  pack_f16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                  pack_f16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
          }
        }
        if (it.part >= 0 && mine) {
          const size_t pi = ((size_t)it.part * kAttnPartRows + row) * REP + hh;
          *reinterpret_cast<float2*>(a.part_ml + pi * 2) = make_float2(mref, l);
        }
        fence_before();   // the next item's first PV overwrites O_t only after this warp's next P arrival
      }
      if (!okd) s_abort = 1;
      gt += nt;
    }
    if (!ok) s_abort = 1;
  } else if (warp < W_MMA + MT) {
    // =============================== every MMA of MMA tile tw, from one thread: O_t += P_t V of a
    // key tile as soon as the warpgroup has written its P, and S_t of a key tile as soon as the
    // tile has landed, its S buffer's previous P has been fed to its PV (issued earlier by this
    // thread: the tensor pipe runs one thread's MMAs in issue order, so the S product cannot
    // overwrite P before the PV has read it) and, for an item's first, its Q tile is written
    const int tw = warp - W_MMA;   // the MMA tile this thread issues for
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(128, KT, false);
      const uint32_t id_pv = idesc_bf16_bmn(128, D);
      uint32_t gt = 0;
      uint32_t ct[MT] = {0, 0}, ci[MT] = {0, 0};   // per MMA tile: key tiles and items taken part in
      bool ok = true;
      for (int ii = blockIdx.x; ii < a.n_items && ok; ii += gridDim.x) {
        const AttnItem it = a.items[ii];
        const int nt = item_tiles(it);
        const int na[MT] = {item_tiles_of(it, 0), item_tiles_of(it, 1)};
        int js[MT] = {0, 0}, jp[MT] = {0, 0};   // next S, next PV (key tiles of the item)
        uint32_t idle = 0;
        unsigned long long t_idle = 0;
        while (jp[tw] < na[tw]) {
          bool prog = false;
          {
            const int t = tw;
            if (jp[t] < js[t]) {   // PV of key tile jp once its P is written
              const uint32_t g = gt + jp[t], c = ct[t] + jp[t];
              const int b = c & 1, st = g % NST;
              if (mbar_test(bar(B_PREADY + 2 * t + b), (c >> 1) & 1)) {
                fence_after();
                const uint32_t vb = smem_u32(sm + OFF_ST + st * ST_BYTES + 16384);
                const uint32_t pa = tmem + TM_S + 128 * t + 64 * b + 32;   // P over the S buffer's high half
#pragma unroll
                for (int k = 0; k < 4; ++k)   // K dimension 64 keys = 4 steps of 16 (8 TMEM columns of P each)
                  umma_ts(tmem + TM_O + 128 * t, pa + 8 * k, desc_mnmajor(vb + k * 2048, 8192), id_pv,
                          (jp[t] | k) != 0);
                umma_commit(bar(B_PVDONE + 2 * t + b));
                umma_commit(bar(B_EMPTY + st));   // the stage's share is released when the PV retires
                ++jp[t];
                prog = true;
              }
            }
            if (js[t] < na[t] && js[t] < jp[t] + 2) {   // S of key tile js into a buffer whose PV is issued
              const uint32_t g = gt + js[t], c = ct[t] + js[t];
              const int b = c & 1, st = g % NST;
              if (mbar_test(bar(B_FULL + st), (g / NST) & 1) &&
                  (js[t] > 0 || mbar_test(bar(B_QREADY + t), ci[t] & 1))) {
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
        }
        for (int t = 0; t < MT; ++t)
          if (na[t] > 0) {
            ct[t] += na[t];
            ++ci[t];
          }
        gt += nt;
      }
      if (!ok) s_abort = 1;
      umma_commit(bar(B_DONE + tw));   // fires once every MMA of this thread has retired
      mbar_wait(bar(B_DONE + tw), 0);
    }
  } else if (warp == W_LOAD) {
    // =============================== loads (lanes issue the boxes; the warp holds page metadata)
    // the grid barrier: every CTA's phase 1 rows are written before the first K box is loaded
    bool ok = true;
    if (lane == 0) {
      const unsigned long long target = a.sync_base + gridDim.x;
      atomicAdd(a.grid_sync, 1ull);
      const unsigned long long t0 = gtimer();
      for (uint32_t i = 0; !s_abort; ++i) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.grid_sync) : "memory");
        if (v >= target) break;
        if ((i & 63) == 63 && gtimer() - t0 > kWaitLimitNs) {
          atomicExch(&g_attn_timeout, 1);
          s_abort = 1;
        }
      }
      ok = !s_abort;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    asm volatile("fence.proxy.async.global;" ::: "memory");   // the TMA loads below read other CTAs' rows
    uint32_t n_ld = 0;   // key tiles issued
    // lane i: metadata of page w0 + i (cur) and of page w0 + 32 + i (nxt, loaded one window ahead)
    int w0 = 0;
    const __nv_bfloat16* vl = static_cast<const __nv_bfloat16*>(a.v_layer);
    for (int ii = blockIdx.x; ii < a.n_items && ok; ii += gridDim.x) {
      const bool first = ii == (int)blockIdx.x;
      const AttnItem it = first ? it_n : a.items[ii];
      const int nt = item_tiles(it);
      auto fetch = [&](int w, int& b, int& p, int& l) { fetch_page(a, it.page1, w + lane, b, p, l); };
      for (int j = 0; j < nt; ++j) {
        const uint32_t gt = n_ld;
        const int s = gt % NST;
        const uint32_t kr = gt / NST;
        const int p0 = it.page0 + 4 * j, np = min(4, it.page1 - p0);
        if (j == 0) {
          w0 = p0;
          if (!first) {   // the first item's window was fetched before phase 1
            fetch(w0, cblk, cpos, clen);
            fetch(w0 + 32, nblk, npos, nlen);
          }
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
        // stage s free once every PV of key tile gt - NST has retired
        if (lane == 0) ok = !s_abort && (kr == 0 || mbar_wait(bar(B_EMPTY + s), (kr - 1) & 1));
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // key positions of the tile (INT_MAX: no key), and its last position (INT_MAX when some
        // slot holds no key: the tile then needs the mask whatever the row)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = 2 * lane + e, q = key >> 4, rr = key & 15;
          const int lq = q == 0 ? len[0] : q == 1 ? len[1] : q == 2 ? len[2] : len[3];
          const int pq = q == 0 ? pos[0] : q == 1 ? pos[1] : q == 2 ? pos[2] : pos[3];
          sPos[s * KT + key] = rr < lq ? pq + rr : INT_MAX;
        }
        bool full[4];
        int n_full = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          full[q] = len[q] == kBlock;
          n_full += full[q];
        }
        if (lane == 0) sTile[s] = n_full == 4 ? pos[3] + kBlock - 1 : INT_MAX;
        const uint32_t kd = smem_u32(sm + OFF_ST + s * ST_BYTES), vd = kd + 16384;
        const bool run = n_full == 4 && blk[1] == blk[0] + 1 && blk[2] == blk[0] + 2 && blk[3] == blk[0] + 3;
        if (n_full < 4) {
          // V of the pages that are not full: rows with a key copied, the others zeroed
          // (4 KB per page: 2 halves x 16 rows x 8 chunks of 16 bytes)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (full[q]) continue;
            const __nv_bfloat16* src = vl + ((size_t)blk[q] * a.G + it.g) * kBlock * D;
            for (int i = lane; i < 256; i += 32) {
              const int h = i >> 7, rr = (i >> 3) & 15, c = i & 7;
              const uint4 v = rr < len[q] ? *reinterpret_cast<const uint4*>(src + rr * D + h * 64 + c * 8)
                                          : make_uint4(0, 0, 0, 0);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(vd + h * 8192 + sw128(q * 16 + rr, c)),
                           "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                           : "memory");
            }
          }
          fence_async_smem();   // the MMAs read these rows through the async proxy
        }
        __syncwarp();
        const uint32_t fb = bar(B_FULL + s);
        // arrives too: the boxes complete the phase (K always 2 x 8 KB; V 2 x 2 KB per full page)
        if (lane == 0) mbar_expect_tx(fb, 16384u + (uint32_t)n_full * 4096u);
        __syncwarp();
        if (lane < 2)   // rotated K: one box of 4 consecutive scratch pages per 64-dim half
          tma_5d(kd + lane * 8192, &a.kmap, 0, lane, 0, it.g, p0, fb);
        if (run) {   // V of 4 consecutive full blocks: one box per half, 8 KB each
          if (lane == 2 || lane == 3) tma_5d(vd + (lane - 2) * 8192, &a.vmap, 0, lane - 2, 0, it.g, blk[0], fb);
        } else if (lane >= 8 && lane < 16) {   // V of one full page per box, 2 KB each
          const int q = (lane - 8) >> 1, h = lane & 1;
          const int bq = q == 0 ? blk[0] : q == 1 ? blk[1] : q == 2 ? blk[2] : blk[3];
          const bool fq = q == 0 ? full[0] : q == 1 ? full[1] : q == 2 ? full[2] : full[3];
          if (fq) tma_5d(vd + h * 8192 + q * 2048, &a.vmap1, 0, h, 0, it.g, bq, fb);
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

// A [n][G][16 rows][128] array of 16-bit elements (`type`: a pool layer of bf16 V, or the fp16
// rotated-K scratch) viewed as (64 dims, 2 halves, 16 rows, G, n): a box is one 64-dim half of
// the 16 rows of one KV head's page in `pages` consecutive entries, landing as [pages][16
// rows][128 B] -- one half of the K-major (K) or MN-major (V) operand of 16 x pages keys.
bool attn_page_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, int n, int G, int pages) {
  auto enc = encode_fn();
  if (!enc || n < 1 || G < 1) return false;
  cuuint64_t dims[5] = {64, 2, (cuuint64_t)kBlock, (cuuint64_t)G, (cuuint64_t)n};
  cuuint64_t strides[4] = {128, (cuuint64_t)D * 2, (cuuint64_t)kBlock * D * 2, (cuuint64_t)G * kBlock * D * 2};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  cuuint32_t box[5] = {64, 1, kBlock, 1, (cuuint32_t)pages};
  return enc(m, type, 5, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool attn_v_map(CUtensorMap* m4, CUtensorMap* m1, const void* v_layer, int pool_blocks, int G) {
  return attn_page_map(m4, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_layer, pool_blocks, G, 4) &&
         attn_page_map(m1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_layer, pool_blocks, G, 1);
}

bool attn_krot_map(CUtensorMap* m, const __half* krot, int n_pages, int G) {
  return attn_page_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, krot, n_pages, G, 4);
}

size_t attention_krot_bytes(int n_pages, int G) { return (size_t)n_pages * G * kBlock * D * sizeof(__half); }

int attention_tc_rows_per_item() { return MT * RB; }

int attention_tc_grid(int n_items) { return std::min(n_items, sm_count()); }

// Grid = min(items, SMs): the planner deals items for exactly this walk. Cooperative (every CTA
// resident: the kernel's grid barrier needs it; the launch fails otherwise) and a programmatic
// dependent of the previous kernel.
void launch_attention_tc(const AttnArgs& a, cudaStream_t st) {
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int smem = SMEM_BYTES + 1024;
  if (dev < 0 || dev >= 64 || !attr[dev]) {
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (dev >= 0 && dev < 64) attr[dev] = true;
  }
  if (a.n_items <= 0) return;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(attention_tc_grid(a.n_items));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, attn_tc_kernel, a);
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
