// Tensor-core paged attention for bf16 KV with head_dim 128 (mma.sync m16n8k16, fp16 operands).
//
// One CTA = one work item: up to 16*RG consecutive query rows of one sequence x the REP
// query heads that share KV head g (GQA) x a run of pages. Warp w owns query head
// g*REP + (w % REP) for the 16 rows of row group w / REP (one MMA M tile), so every K/V
// tile staged in shared memory feeds RG*REP warps. KV moves in tiles of 64 keys (4 pages):
//   * K: cp.async into a raw buffer one tile ahead, then rotated by RoPE at each key's
//     absolute position, shared -> shared, into the double-buffered operand tile (MEPIC
//     abstract: K is kept without positional encoding and RoPE is fused into attention).
//     For a key at row r of a page that starts at position P, cos/sin((P + r) theta) is
//     composed from the table row of P (one per page, staged by cp.async) and the row of
//     r (resident), so a tile reads 4 table rows instead of 64.
//   * V: cp.async into a raw buffer, converted to fp16 in the same pass.
//   Operands are fp16 (bf16 K/V values are exact in fp16; q arrives in fp32 and is rounded
//   once, after RoPE); S, the softmax and O are fp32; the output is fp16.
//   * page metadata (block, start, length) is cached in shared memory in windows of 512
//     pages, so no global load sits in front of the KV loads.
// S = Q K^T and O += P V run on mma.sync with fp32 accumulators; the online softmax
// lives in registers (row max/sum by quad shuffles). Keys after the query's position,
// padding rows of ragged pages and pages past the item's range are masked. Items that
// cover part of a row block's pages write unnormalized partials (o, m, l) that the merge
// kernel of k_attn.cu combines.
#include <climits>

#include "pic_internal.h"

namespace pic {

void launch_attention_simt(const AttnArgs& a, cudaStream_t st);

namespace {

constexpr int D = 128;
constexpr int KT = 64;                    // keys per tile
constexpr int TILE_BYTES = KT * D * 2;    // 16 KB
constexpr int WIN = 512;                  // pages of metadata cached at once
constexpr float kLog2e = 1.4426950408889634f;

// byte offset of 16-byte chunk `c` (0..15) of row `r` in a [rows][128] bf16 tile, XOR-swizzled
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// rotate 8 dims (i) and their partners (i + 64) by the composed angle, times `scale`, to fp16
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

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(b[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}

template <int REP, int RG>
__global__ void __launch_bounds__(REP * RG * 32) attn_mma_kernel(AttnArgs a) {
  constexpr int NW = REP * RG, NT = NW * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem;                                   // [2][KT][D] rotated K (Q staging at start)
  uint8_t* sKr = sK + 2 * TILE_BYTES;                   // [KT][D] raw (bf16) K of the next tile
  uint8_t* sVr = sKr + TILE_BYTES;                      // [KT][D] raw (bf16) V of the next tile
  uint8_t* sV = sVr + TILE_BYTES;                       // [2][KT][D] fp16 V operand
  float2* sLo = reinterpret_cast<float2*>(sV + 2 * TILE_BYTES);   // [16][64] cos/sin of p = 0..15
  float2* sPg = sLo + 16 * 64;                                     // [2][4][64] cos/sin of page starts
  int* sBlk = reinterpret_cast<int*>(sPg + 2 * 4 * 64);            // [WIN] page metadata window
  int* sPp = sBlk + WIN;
  int* sPl = sPp + WIN;
  int* sPos = sPl + WIN;                                           // [2][KT] key positions (INT_MAX = masked)
  const uint32_t sK_u = (uint32_t)__cvta_generic_to_shared(sK);
  const uint32_t sKr_u = (uint32_t)__cvta_generic_to_shared(sKr);
  const uint32_t sVr_u = (uint32_t)__cvta_generic_to_shared(sVr);
  const uint32_t sPg_u = (uint32_t)__cvta_generic_to_shared(sPg);

  const AttnItem it = a.items[blockIdx.x];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G;
  const __nv_bfloat16* Kl = (const __nv_bfloat16*)a.k_layer;
  const __nv_bfloat16* Vl = (const __nv_bfloat16*)a.v_layer;
  const float* Q = a.q;
  const int npages = it.page1 - it.page0;
  const int ntiles = (npages + 3) / 4;

  auto load_meta = [&](int win0) {
    for (int i = tid; i < WIN; i += NT) {
      const int pg = it.page0 + win0 + i;
      if (pg < it.page1) {
        sBlk[i] = a.page_block[pg];
        sPp[i] = a.page_pos[pg];
        sPl[i] = a.page_len[pg];
      }
    }
  };
  for (int i = tid; i < 16 * 64; i += NT) sLo[i] = a.rope_cs[i];
  int win = 0;
  load_meta(0);
  __syncthreads();

  // ---- Q: rotate at each row's position, scale into log2 units, stage for ldmatrix
  const float qscale = rsqrtf((float)D) * kLog2e;
  for (int i = tid; i < NW * 16 * 8; i += NT) {
    const int w = i / 128, r16 = (i / 8) % 16, c = i % 8;
    const int r = (w / REP) * 16 + r16, qh = w % REP;
    uint4 y1 = make_uint4(0, 0, 0, 0), y2 = y1;
    if (r < it.nrows) {
      const int t = it.row0 + r, h = it.g * REP + qh, p = a.q_pos[t];
      const float* src = Q + ((size_t)t * a.H + h) * D;
      float v1[8], v2[8];
      *reinterpret_cast<float4*>(v1) = *reinterpret_cast<const float4*>(src + 8 * c);
      *reinterpret_cast<float4*>(v1 + 4) = *reinterpret_cast<const float4*>(src + 8 * c + 4);
      *reinterpret_cast<float4*>(v2) = *reinterpret_cast<const float4*>(src + 64 + 8 * c);
      *reinterpret_cast<float4*>(v2 + 4) = *reinterpret_cast<const float4*>(src + 64 + 8 * c + 4);
      rope8(v1, v2, a.rope_cs + (size_t)(p & ~15) * 64 + 8 * c, sLo + (p & 15) * 64 + 8 * c, qscale, y1, y2);
    }
    uint8_t* base = sK + w * 16 * D * 2;
    *reinterpret_cast<uint4*>(base + swz(r16, c)) = y1;
    *reinterpret_cast<uint4*>(base + swz(r16, c + 8)) = y2;
  }
  __syncthreads();
  const int rg = warp / REP, hh = warp % REP;
  const bool active = rg * 16 < it.nrows;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int row0 = rg * 16 + g8, row1 = row0 + 8;
  const int qp0 = row0 < it.nrows ? a.q_pos[it.row0 + row0] : -1;
  const int qp1 = row1 < it.nrows ? a.q_pos[it.row0 + row1] : -1;
  uint32_t qf[8][4];
  {
    const uint32_t qb = sK_u + warp * 16 * D * 2;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int m = lane >> 3, row = (lane & 7) + 8 * (m & 1), c = 2 * ks + (m >> 1);
      ldsm_x4(qb + swz(row, c), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  }
  __syncthreads();  // the Q staging area becomes the K operand buffers

  // ---- tile loaders (page metadata relative to the current window)
  auto issue_loads = [&](int tile, int buf) {
    const int pbase = tile * 4 - win;  // window index of the tile's first page
    for (int task = tid; task < KT * 16; task += NT) {
      const int key = task / 16, c = task % 16;
      const int pi = pbase + key / 16, r = key % 16;
      const bool valid = tile * 4 + key / 16 < npages && r < sPl[pi];
      const uint32_t off = swz(key, c);
      if (valid) {
        const size_t src = (((size_t)sBlk[pi] * G + it.g) * kBlock + r) * D + 8 * c;
        cp_async16(sKr_u + off, Kl + src);
        cp_async16(sVr_u + off, Vl + src);
      }
    }
    for (int i = tid; i < 4 * 32; i += NT) {   // 4 page-start RoPE rows of 512 B
      const int pg = i / 32, c = i % 32;
      if (tile * 4 + pg < npages)
        cp_async16(sPg_u + (uint32_t)((buf * 4 + pg) * 64 * sizeof(float2) + c * 16),
                   a.rope_cs + (size_t)sPp[pbase + pg] * 64 + c * 2);
    }
  };
  // raw bf16 K and V of a tile -> fp16 operands: K rotated at each key's position, V converted;
  // padding and out-of-range keys become zeros with position INT_MAX (masked)
  auto prepare_kv = [&](int tile, int buf) {
    const int pbase = tile * 4 - win;
    for (int task = tid; task < KT * 8; task += NT) {
      const int key = task / 8, c = task % 8;
      const int pi = pbase + key / 16, r = key % 16;
      const bool valid = tile * 4 + key / 16 < npages && r < sPl[pi];
      uint4 k1 = make_uint4(0, 0, 0, 0), k2 = k1, v1 = k1, v2 = k1;
      if (valid) {
        float a1[8], a2[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sKr + swz(key, c)), a1);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sKr + swz(key, c + 8)), a2);
        rope8(a1, a2, sPg + (buf * 4 + key / 16) * 64 + 8 * c, sLo + r * 64 + 8 * c, 1.f, k1, k2);
        float b1[8], b2[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sVr + swz(key, c)), b1);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sVr + swz(key, c + 8)), b2);
        __half h1[8], h2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          h1[e] = __float2half_rn(b1[e]);
          h2[e] = __float2half_rn(b2[e]);
        }
        v1 = *reinterpret_cast<uint4*>(h1);
        v2 = *reinterpret_cast<uint4*>(h2);
      }
      uint8_t* kb_ = sK + buf * TILE_BYTES;
      uint8_t* vb_ = sV + buf * TILE_BYTES;
      *reinterpret_cast<uint4*>(kb_ + swz(key, c)) = k1;
      *reinterpret_cast<uint4*>(kb_ + swz(key, c + 8)) = k2;
      *reinterpret_cast<uint4*>(vb_ + swz(key, c)) = v1;
      *reinterpret_cast<uint4*>(vb_ + swz(key, c + 8)) = v2;
      if (c == 0) sPos[buf * KT + key] = valid ? sPp[pi] + r : INT_MAX;
    }
  };

  if (ntiles > 0) issue_loads(0, 0);
  cp_async_wait_all();
  __syncthreads();
  if (ntiles > 0) prepare_kv(0, 0);
  __syncthreads();

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int tile = 0; tile < ntiles; ++tile) {
    const int cur = tile & 1, nxt = cur ^ 1;
    const bool has_next = tile + 1 < ntiles;
    if (has_next) {
      const int w1 = ((tile + 1) * 4 / WIN) * WIN;
      if (w1 != win) {  // the next tile starts a new metadata window (same for every thread)
        __syncthreads();
        win = w1;
        load_meta(win);
        __syncthreads();
      }
      issue_loads(tile + 1, nxt);
    }
    if (active) {
      // S = Q K^T over 64 keys
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
      const uint32_t kb = sK_u + cur * TILE_BYTES;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          const int m = lane >> 3, key = 8 * j + (lane & 7) + 8 * (m >> 1), c = 2 * ks + (m & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz(key, c), b0, b1, b2, b3);
          mma16816(s[j], qf[ks], b0, b1);
          mma16816(s[j + 1], qf[ks], b2, b3);
        }
      }
      // mask + online softmax (rows row0 and row1; this thread holds keys 8j+2t4, +1)
      const int* kp = sPos + cur * KT;
      float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int p = kp[8 * j + 2 * t4 + e];
          if (p > qp0) s[j][e] = -INFINITY;
          if (p > qp1) s[j][2 + e] = -INFINITY;
          tm0 = fmaxf(tm0, s[j][e]);
          tm1 = fmaxf(tm1, s[j][2 + e]);
        }
      }
      tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, 1));
      tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, 2));
      tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, 1));
      tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, 2));
      const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float corr0 = exp2f(m0 - ref0), corr1 = exp2f(m1 - ref1);
      m0 = mn0;
      m1 = mn1;
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pf[4][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p0 = exp2f(s[j][0] - ref0), p1 = exp2f(s[j][1] - ref0);
        const float p2 = exp2f(s[j][2] - ref1), p3 = exp2f(s[j][3] - ref1);
        rs0 += p0 + p1;
        rs1 += p2 + p3;
        pf[j >> 1][(j & 1) * 2 + 0] = pack_h2(p0, p1);
        pf[j >> 1][(j & 1) * 2 + 1] = pack_h2(p2, p3);
      }
      l0 = l0 * corr0 + rs0;
      l1 = l1 * corr1 + rs1;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= corr0;
        o[i][1] *= corr0;
        o[i][2] *= corr1;
        o[i][3] *= corr1;
      }
      // O += P V
      const uint32_t vb = (uint32_t)__cvta_generic_to_shared(sV) + cur * TILE_BYTES;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // A fragment of P for keys 16kk..16kk+15: {row0 k0-7, row1 k0-7, row0 k8-15, row1 k8-15}
        const uint32_t af[4] = {pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3]};
#pragma unroll
        for (int dn = 0; dn < 16; dn += 2) {
          const int m = lane >> 3, key = 16 * kk + (lane & 7) + 8 * (m & 1), c = dn + (m >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + swz(key, c), b0, b1, b2, b3);
          mma16816(o[dn], af, b0, b1);
          mma16816(o[dn + 1], af, b2, b3);
        }
      }
    }
    cp_async_wait_all();   // raw K and V and the page RoPE rows of the next tile have landed
    __syncthreads();
    if (has_next) prepare_kv(tile + 1, nxt);
    __syncthreads();
  }

  if (!active) return;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const int h = it.g * REP + hh;
  if (it.part < 0) {
    __half* out = (__half*)a.out;
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) {
      const int dcol = 8 * dn + 2 * t4;
      if (row0 < it.nrows)
        *reinterpret_cast<uint32_t*>(out + ((size_t)(it.row0 + row0) * a.H + h) * D + dcol) =
            pack_h2(o[dn][0] * i0, o[dn][1] * i0);
      if (row1 < it.nrows)
        *reinterpret_cast<uint32_t*>(out + ((size_t)(it.row0 + row1) * a.H + h) * D + dcol) =
            pack_h2(o[dn][2] * i1, o[dn][3] * i1);
    }
  } else {
    const size_t p0 = ((size_t)it.part * kAttnPartRows + row0) * REP + hh;
    const size_t p1 = ((size_t)it.part * kAttnPartRows + row1) * REP + hh;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) {
      const int dcol = 8 * dn + 2 * t4;
      *reinterpret_cast<float2*>(a.part_o + p0 * D + dcol) = make_float2(o[dn][0], o[dn][1]);
      *reinterpret_cast<float2*>(a.part_o + p1 * D + dcol) = make_float2(o[dn][2], o[dn][3]);
    }
    if (t4 == 0) {
      a.part_ml[p0 * 2] = m0;
      a.part_ml[p0 * 2 + 1] = l0;
      a.part_ml[p1 * 2] = m1;
      a.part_ml[p1 * 2 + 1] = l1;
    }
  }
}

template <int REP, int RG>
void launch_rep(const AttnArgs& a, cudaStream_t st) {
  constexpr int NW = REP * RG;
  static_assert(NW * 16 * D * 2 <= 2 * TILE_BYTES, "Q staging must fit the K operand buffers");
  const size_t smem = 6 * TILE_BYTES + (16 + 2 * 4) * 64 * sizeof(float2) + (3 * WIN + 2 * KT) * sizeof(int);
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr[dev]) {
    cudaFuncSetAttribute(attn_mma_kernel<REP, RG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (dev >= 0 && dev < 64) attr[dev] = true;
  }
  attn_mma_kernel<REP, RG><<<a.n_items, NW * 32, smem, st>>>(a);
}

}  // namespace

void launch_attention_mma(const AttnArgs& a, cudaStream_t st) {
  const int rep = a.H / a.G;
  if (a.n_items > 0) {
    switch (rep) {   // rows per item: 32 (two row groups) for rep <= 4, 16 for rep 8
      case 1: launch_rep<1, 2>(a, st); break;
      case 2: launch_rep<2, 2>(a, st); break;
      case 4: launch_rep<4, 2>(a, st); break;
      case 8: launch_rep<8, 1>(a, st); break;
      default: launch_attention_simt(a, st); return;
    }
  }
  if (a.n_combines > 0) {
    AttnArgs b = a;
    b.n_items = 0;  // merge only
    launch_attention_simt(b, st);
  }
}

}  // namespace pic
