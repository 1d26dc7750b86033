// C ABI: model and paged store, compile, link (LegoLink-k), release, kernel-level calls.
//
// Host-side work here is the integer bookkeeping of the method: the block allocator
// (lowest free id first, all-or-nothing), chunk and request tables with reference
// counts, the selected-row list, the per-request page tables and the slot mapping.
// Every arithmetic step of the forward pass runs in the library's CUDA kernels.
//
// Method sources: "EPIC: Efficient Position-Independent Caching for Serving Large
// Language Models" (summary page: summary line, Approach, Measured effects table) for
// compile/link, LegoLink-k and LegoLink-0; "MEPIC: Memory Efficient Position
// Independent Caching for LLM Serving" (abstract) for page-aligned chunk KV, the
// request-specific first block, shared remaining blocks and RoPE fused in attention.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <list>
#include <map>
#include <memory>
#include <set>

#include "pic_internal.h"

namespace pic {

static thread_local std::string g_last_error;
void set_error(const std::string& msg) { g_last_error = msg; }
pic_status fail(pic_status s, const std::string& msg) {
  g_last_error = msg;
  if (s == PIC_ERR_CUDA) (void)cudaGetLastError();  // do not leak a non-sticky error into later calls
  return s;
}

}  // namespace pic

using namespace pic;

struct pic_model {
  pic_model_config cfg{};
  const void* embed = nullptr;
  const void* lm_head = nullptr;
  const float* final_norm = nullptr;
  std::vector<const float*> attn_norm, mlp_norm;
  std::vector<const void*> wqkv, wo, wgu, wdown;
  int device = 0;
  int num_sms = 0;
  // bf16: projection matrices repacked once into the tcgen05 tile layout (library-owned)
  void* packed = nullptr;
  std::vector<const void*> pqkv, po, pgu, pdown;
  const void* plm = nullptr;
  int qkv_dim() const { return (cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim; }
  ~pic_model() { cudaFree(packed); }
};

namespace {

struct Chunk {
  std::vector<int32_t> tokens;
  std::vector<int32_t> blocks;
  int refs = 1;
  int n_dummy = 0;
  bool cached = false;   // from pic_compile_cached: indexed by content, kept resident at refs 0
  uint64_t key = 0;      // content hash (cached chunks)
};

// FNV-1a over (n_dummy, length, token ids): the bucket of a chunk's content in the store's
// index (a hit is confirmed by comparing the tokens themselves).
uint64_t content_key(const int32_t* tokens, int n, int n_dummy) {
  uint64_t h = 1469598103934665603ull;
  auto mix = [&](uint32_t v) {
    for (int b = 0; b < 4; ++b) {
      h ^= (v >> (8 * b)) & 0xffu;
      h *= 1099511628211ull;
    }
  };
  mix((uint32_t)n_dummy);
  mix((uint32_t)n);
  for (int i = 0; i < n; ++i) mix((uint32_t)tokens[i]);
  return h;
}

struct Request {
  std::vector<int32_t> chunk_ids;
  std::vector<int32_t> selected, slots, page_table, page_pos, page_len, private_blocks;
};

// One forward pass over a set of rows grouped in sequences (compile: chunks; link: requests).
struct Batch {
  std::vector<int> tok, pos, slot, out_row, lg_row;
  std::vector<int> pblk, ppos, plen;
  std::vector<int> seq_row_begin, seq_row_end, seq_page_begin, seq_page_end;
  std::vector<int> copy_pairs;
  int n_hidden = 0, n_lg = 0;
  bool compile = false;
  int rows() const { return (int)tok.size(); }
  void begin_seq() {
    seq_row_begin.push_back(rows());
    seq_page_begin.push_back((int)pblk.size());
  }
  void end_seq() {
    seq_row_end.push_back(rows());
    seq_page_end.push_back((int)pblk.size());
  }
  void row(int t, int p, int s) {
    tok.push_back(t);
    pos.push_back(p);
    slot.push_back(s);
    out_row.push_back(-1);
    lg_row.push_back(-1);
  }
  void page(int b, int p, int l) {
    pblk.push_back(b);
    ppos.push_back(p);
    plen.push_back(l);
  }
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

struct pic_store {
  pic_model* m = nullptr;
  pic_store_config cfg{};
  void* k_pool = nullptr;
  void* v_pool = nullptr;
  std::set<int32_t> free;
  std::map<int32_t, Chunk> chunks;
  // content-addressed reuse (pic_compile_cached): content hash -> chunk id, and the cached
  // chunks nothing references, least recently released first (evicted in that order)
  std::multimap<uint64_t, int32_t> cache_index;
  std::list<int32_t> lru;
  int64_t cache_hits = 0, cache_misses = 0, cache_evictions = 0;
  std::map<int32_t, Request> requests;
  int32_t next_chunk = 1, next_request = 1;

  // library-owned device workspace (one allocation)
  char* ws = nullptr;
  float* h = nullptr;
  void* x = nullptr;
  float* q = nullptr;        // [max_rows][H*D] fp32 pre-RoPE, or fp16 rotated (tensor-core attention)
  void* attn = nullptr;
  void* act = nullptr;
  void* lm_x = nullptr;
  float* qkv_acc = nullptr;  // [max_rows][(H+2G)D] fp32, the QKV GEMM's result
  float* gu_acc = nullptr;   // [max_rows][2F] fp32, the gate/up GEMM's result
  // tcgen05 GEMMs that start their output at zero themselves publish each zeroed tile here as
  // the launch's epoch (device ints, zero at creation; epochs start at 1)
  int* tile_ready = nullptr;
  size_t tile_ready_cap = 0;
  uint32_t gemm_epoch = 0;
  uint32_t next_epoch() {
    if (++gemm_epoch == 0) ++gemm_epoch;
    return gemm_epoch;
  }
  float* att_o = nullptr;
  float* att_ml = nullptr;
  int att_parts_cap = 0;
  int32_t* meta_d = nullptr;
  size_t meta_cap = 0;  // int32 elements
  float2* rope_cs = nullptr;
  std::vector<CUtensorMap> v_maps;   // per layer: V pool boxes of 4 blocks, of 1 block; built on first use
  // rotated K of every page of a forward, one layer at a time (tensor-core attention): grown
  // on first need to the largest page count seen
  __half* krot = nullptr;
  int krot_pages = 0;
  // grid-barrier counter of the tensor-core attention (workspace, zero at creation) and the
  // number of CTA arrivals every earlier launch adds to it
  unsigned long long* att_sync = nullptr;
  unsigned long long att_sync_total = 0;
  // query-key logits of a dynamic-selection pass: grown on first need to the largest pass seen
  float* sel_logits = nullptr;
  size_t sel_logits_cap = 0;
  int32_t* meta_h = nullptr;  // pinned staging
  cudaEvent_t meta_ev = nullptr;
  bool meta_ev_pending = false;

  // profiling: event pairs around launches while enabled; launch counter always on
  struct ProfRec {
    int cls;
    cudaEvent_t a, b;
    double bytes, flops;
    int launches;
  };
  bool prof_on = false;
  std::vector<ProfRec> prof;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  int64_t launches = 0;

  cudaEvent_t next_event() {
    if (ev_used == ev_pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      ev_pool.push_back(e);
    }
    return ev_pool[ev_used++];
  }

  int scratch_block() const { return cfg.num_blocks; }
  int blocks_total() const { return cfg.num_blocks + 1; }
  size_t block_bytes() const {
    const auto& c = m->cfg;
    return (size_t)c.n_kv_heads * kBlock * c.head_dim * dtype_size(c.dtype);
  }
  size_t layer_bytes() const { return block_bytes() * blocks_total(); }
  void* k_layer(int l) const { return (char*)k_pool + layer_bytes() * l; }
  void* v_layer(int l) const { return (char*)v_pool + layer_bytes() * l; }
  int att_blocks_cap() const { return cfg.max_rows / kBlock + cfg.max_requests + 2; }

  std::vector<int32_t> take(int n) {
    std::vector<int32_t> ids;
    auto it = free.begin();
    for (int i = 0; i < n; ++i) ids.push_back(*it++);
    for (int32_t b : ids) free.erase(b);
    return ids;
  }
  void give(const std::vector<int32_t>& ids) { free.insert(ids.begin(), ids.end()); }

  // A chunk handle the caller may use: alive and referenced (a released cached chunk stays
  // resident for reuse but its old handle is gone).
  Chunk* live_chunk(int32_t id) {
    auto it = chunks.find(id);
    return it == chunks.end() || it->second.refs < 1 ? nullptr : &it->second;
  }
  // The chunk's last reference is gone: a cached chunk stays resident (evictable), any other
  // returns its blocks.
  void retire(int32_t id) {
    auto it = chunks.find(id);
    if (it == chunks.end()) return;
    if (it->second.cached) {
      lru.push_back(id);
      return;
    }
    give(it->second.blocks);
    chunks.erase(it);
  }
  void evict_front() {
    const int32_t id = lru.front();
    lru.pop_front();
    auto it = chunks.find(id);
    auto range = cache_index.equal_range(it->second.key);
    for (auto i = range.first; i != range.second; ++i)
      if (i->second == id) {
        cache_index.erase(i);
        break;
      }
    give(it->second.blocks);
    chunks.erase(it);
    ++cache_evictions;
  }
  // Makes `need` blocks free, evicting unreferenced cached chunks least recently released
  // first; evicts nothing and returns false when even evicting all of them is not enough.
  bool reserve(int need) {
    size_t avail = free.size();
    for (int32_t id : lru) avail += chunks[id].blocks.size();
    if ((size_t)std::max(0, need) > avail) return false;
    while ((int)free.size() < need) evict_front();
    return true;
  }
  // A cached chunk with the same content and dummy prefix (0 when none).
  int32_t find_cached(uint64_t key, const int32_t* tokens, int n, int n_dummy) {
    auto range = cache_index.equal_range(key);
    for (auto i = range.first; i != range.second; ++i) {
      const Chunk& c = chunks[i->second];
      if (c.n_dummy == n_dummy && (int)c.tokens.size() == n && std::equal(c.tokens.begin(), c.tokens.end(), tokens))
        return i->second;
    }
    return 0;
  }
  // One more reference to a chunk (taking it off the eviction list if it was there).
  void ref(int32_t id) {
    Chunk& c = chunks[id];
    if (c.refs == 0) lru.remove(id);
    ++c.refs;
  }
};

namespace {

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Y[T][N] += X . W^T (fp32 Y accumulated in place), or Y = X . W^T when `overwrite`; Wp: the
// packed copy of W, if any. A packed GEMM that overwrites zeroes Y's tiles itself; otherwise Y
// is cleared by a kernel first.
pic_status gemm(pic_store* s, const void* W, const void* Wp, const void* X, float* Y, int N, int K, int T,
                cudaStream_t st, bool overwrite) {
  if (Wp) {
    if (overwrite && tc_gemm_tiles(N, T) <= s->tile_ready_cap)   // model weights: fixed since creation
      return tc_gemm_run_packed(Wp, X, Y, N, K, T, st, true, s->tile_ready, s->next_epoch());
    if (overwrite) launch_zero(Y, (size_t)T * N, st);
    return tc_gemm_run_packed(Wp, X, Y, N, K, T, st, true);
  }
  if (overwrite) launch_zero(Y, (size_t)T * N, st);
  launch_gemm_simt(s->m->cfg.dtype, s->m->cfg.dtype == PIC_BF16, W, X, Y, N, K, T, 1, st);
  return PIC_OK;
}

// Brackets one step (one or more kernel launches) with profiling events when enabled.
struct Rec {
  pic_store* s;
  cudaStream_t st;
  pic_store::ProfRec r{};
  Rec(pic_store* s_, cudaStream_t st_, int cls, double bytes, double flops, int n_launch) : s(s_), st(st_) {
    s->launches += n_launch;
    if (!s->prof_on) return;
    r.cls = cls;
    r.bytes = bytes;
    r.flops = flops;
    r.launches = n_launch;
    r.a = s->next_event();
    r.b = s->next_event();
    if (r.a) cudaEventRecord(r.a, st);
  }
  ~Rec() {
    if (!s->prof_on || !r.a || !r.b) return;
    cudaEventRecord(r.b, st);
    s->prof.push_back(r);
  }
};

// Uploads the batch metadata and runs embedding, every layer, and (link) the LM head.
pic_status run_forward_impl(pic_store* s, const Batch& b, float* hidden_out, float* logits_out, cudaStream_t st) {
  const pic_model_config& c = s->m->cfg;
  const int T = b.rows();
  const int dt = c.dtype;
  const int H = c.n_heads, G = c.n_kv_heads, D = c.head_dim, d = c.d_model, F = c.ffn_dim;
  if (T > s->cfg.max_rows) return fail(PIC_ERR_CAPACITY, "rows exceed max_rows");
  if (b.n_lg > s->cfg.max_logit_rows) return fail(PIC_ERR_CAPACITY, "logit rows exceed max_logit_rows");
  if ((int)b.seq_row_begin.size() > s->cfg.max_requests + 1)
    return fail(PIC_ERR_CAPACITY, "sequences exceed max_requests");

  // attention work plan
  AttnPlanInput pin;
  pin.seq_row_begin = b.seq_row_begin;
  pin.seq_row_end = b.seq_row_end;
  pin.seq_page_begin = b.seq_page_begin;
  pin.seq_page_end = b.seq_page_end;
  pin.row_pos = &b.pos;
  pin.page_pos = &b.ppos;
  pin.G = G;
  pin.num_sms = s->m->num_sms;
  pin.rows_per_block = attention_rows_per_block(dt, D, H / G);
  pin.persistent = attention_persistent(dt, D, H / G);
  std::vector<AttnItem> items;
  std::vector<AttnCombine> combs;
  int n_parts = 0;
  plan_attention(pin, items, combs, n_parts);
  if (n_parts > s->att_parts_cap) return fail(PIC_ERR_CAPACITY, "attention split plan exceeds workspace");

  // pack metadata: tok pos slot out lg | pblk ppos plen | copies | items | combines
  const size_t P = b.pblk.size(), NC = b.copy_pairs.size();
  const size_t n_int = 5 * (size_t)T + 3 * P + NC + items.size() * kAttnItemInts + combs.size() * 5;
  if (n_int > s->meta_cap) return fail(PIC_ERR_CAPACITY, "metadata exceeds workspace");
  if (s->meta_ev_pending) {
    PIC_CUDA(cudaEventSynchronize(s->meta_ev));
    s->meta_ev_pending = false;
  }
  int32_t* hp = s->meta_h;
  size_t o = 0;
  auto put = [&](const void* src, size_t n) {
    if (n) std::memcpy(hp + o, src, n * 4);
    const size_t at = o;
    o += n;
    return s->meta_d + at;
  };
  const int* d_tok = put(b.tok.data(), T);
  const int* d_pos = put(b.pos.data(), T);
  const int* d_slot = put(b.slot.data(), T);
  const int* d_out = put(b.out_row.data(), T);
  const int* d_lg = put(b.lg_row.data(), T);
  const int* d_pblk = put(b.pblk.data(), P);
  const int* d_ppos = put(b.ppos.data(), P);
  const int* d_plen = put(b.plen.data(), P);
  const int* d_copy = put(b.copy_pairs.data(), NC);
  const AttnItem* d_items = (const AttnItem*)put(items.data(), items.size() * kAttnItemInts);
  const AttnCombine* d_combs = (const AttnCombine*)put(combs.data(), combs.size() * 5);
  PIC_CUDA(cudaMemcpyAsync(s->meta_d, hp, o * 4, cudaMemcpyHostToDevice, st));
  PIC_CUDA(cudaEventRecord(s->meta_ev, st));
  s->meta_ev_pending = true;

  const size_t es = dtype_size(dt);
  const double dT = T, dd = d, dHD = (double)H * D, dF = F, dQKV = s->m->qkv_dim();
  // copy-on-write of the request-private first blocks (all layers, K and V)
  if (NC) {
    Rec r(s, st, PIC_PROF_COPY, (double)NC / 2 * 2 * 2 * c.n_layers * s->block_bytes(), 0, 1);
    launch_copy_blocks((int)NC / 2, d_copy, c.n_layers, s->blocks_total(), s->block_bytes(), s->k_pool, s->v_pool, st);
  }

  // attention work per layer: KV pages read once, queries and outputs once
  double att_kv_bytes = 0, att_pairs = 0;
  for (size_t q = 0; q < b.seq_row_begin.size(); ++q) {
    int last = -1;
    for (int r = b.seq_row_begin[q]; r < b.seq_row_end[q]; ++r) last = std::max(last, b.pos[r]);
    for (int p = b.seq_page_begin[q]; p < b.seq_page_end[q]; ++p)
      if (b.ppos[p] <= last) att_kv_bytes += (double)b.plen[p] * G * D * 2 * es;
    // visible keys of a row: full pages before its page + the visible part of its page
    const int p0 = b.seq_page_begin[q], p1 = b.seq_page_end[q];
    std::vector<double> cum(p1 - p0 + 1, 0.0);
    for (int p = p0; p < p1; ++p) cum[p - p0 + 1] = cum[p - p0] + b.plen[p];
    for (int r = b.seq_row_begin[q]; r < b.seq_row_end[q]; ++r) {
      const int p = (int)(std::upper_bound(b.ppos.begin() + p0, b.ppos.begin() + p1, b.pos[r]) - b.ppos.begin()) - 1;
      if (p >= p0) att_pairs += cum[p - p0] + std::min(b.plen[p], b.pos[r] - b.ppos[p] + 1);
    }
  }
  const double att_bytes = att_kv_bytes + 2 * dT * dHD * es;
  const double att_flops = att_pairs * H * D * 4.0;
  const int att_launches = 1 + (combs.empty() ? 0 : 1);
  // the K rotation inside the tensor-core attention: every page's K read, rotated K written
  const double rot_bytes = 2.0 * (double)P * G * kBlock * D * 2;

  AttnArgs aa{};
  const bool att_tc = attention_persistent(dt, D, H / G);
  const int n_pages = (int)P;
  if (att_tc) {
    if (s->v_maps.empty()) {
      s->v_maps.resize(2 * (size_t)c.n_layers);
      for (int l = 0; l < c.n_layers; ++l)
        if (!attn_v_map(&s->v_maps[2 * l], &s->v_maps[2 * l + 1], s->v_layer(l), s->blocks_total(), G)) {
          s->v_maps.clear();
          return fail(PIC_ERR_CUDA, "cuTensorMapEncodeTiled failed for the V pools");
        }
    }
    if (n_pages > s->krot_pages) {
      // cudaFree waits for the kernels still reading the old scratch
      const int want = std::max(n_pages, s->krot_pages + s->krot_pages / 4);
      __half* fresh = nullptr;
      PIC_CUDA(cudaFree(s->krot));
      s->krot = nullptr;
      s->krot_pages = 0;
      PIC_CUDA(cudaMalloc(&fresh, attention_krot_bytes(want, G)));
      s->krot = fresh;
      s->krot_pages = want;
    }
    if (!attn_krot_map(&aa.kmap, s->krot, std::max(1, n_pages), G))
      return fail(PIC_ERR_CUDA, "cuTensorMapEncodeTiled failed for the rotated-K scratch");
    aa.krot = s->krot;
    aa.n_pages = n_pages;
    aa.grid_sync = s->att_sync;
    aa.q16 = (const __half*)s->q;   // written rotated and scaled by the QKV epilogue
  }
  aa.dtype = dt;
  aa.rb = pin.rows_per_block;
  aa.H = H;
  aa.G = G;
  aa.D = D;
  aa.q = s->q;
  aa.q_pos = d_pos;
  aa.page_block = d_pblk;
  aa.page_pos = d_ppos;
  aa.page_len = d_plen;
  aa.rope_cs = s->rope_cs;
  aa.out = s->attn;
  aa.part_o = s->att_o;
  aa.part_ml = s->att_ml;
  aa.items = d_items;
  aa.n_items = (int)items.size();
  aa.combines = d_combs;
  aa.n_combines = (int)combs.size();

  const int qkv = s->m->qkv_dim();
  auto gemm_bytes = [&](double N, double K, double rows) { return N * K * es + rows * K * es + rows * N * 4; };
  // The QKV, gate/up and LM-head GEMMs write fresh results (a tcgen05 GEMM zeroes its output
  // tiles itself before its split-K reduce-adds land; a SIMT GEMM's output is cleared by a kernel
  // first); the O and down projections add straight into the residual stream h. Every kernel of
  // the forward is a programmatic dependent launch of the one before it.
  auto pk = [&](const std::vector<const void*>& v, int l) -> const void* { return v.empty() ? nullptr : v[l]; };
  auto run_gemm = [&](const void* W, const void* Wp, const void* X, float* Y, int N, int K, int rows, bool overwrite,
                      int cls = PIC_PROF_GEMM) {
    const bool zero_kernel = overwrite && !(Wp && tc_gemm_tiles(N, rows) <= s->tile_ready_cap);
    Rec r(s, st, cls, gemm_bytes(N, K, rows) + (overwrite ? (double)rows * N * 4 : 0), 2.0 * N * K * rows,
          1 + (zero_kernel ? 1 : 0));
    return gemm(s, W, Wp, X, Y, N, K, rows, st, overwrite);
  };
  {
    Rec r(s, st, PIC_PROF_ROWWISE, dT * dd * (es + 4 + es) + dT * 4, 0, 1);
    launch_embed_norm(dt, T, d, s->m->embed, d_tok, s->m->attn_norm[0], c.rms_eps, s->h, s->x, st);
  }
  for (int l = 0; l < c.n_layers; ++l) {
    pic_status e;
    if ((e = run_gemm(s->m->wqkv[l], pk(s->m->pqkv, l), s->x, s->qkv_acc, qkv, d, T, true)) != PIC_OK) return e;
    {
      Rec r(s, st, PIC_PROF_ROWWISE, dT * dQKV * (4 + es), 0, 1);
      launch_qkv_epilogue(dt, T, H, G, D, s->qkv_acc, s->q, d_slot, s->k_layer(l), s->v_layer(l), d_pos, s->rope_cs,
                          att_tc ? (__half*)s->q : nullptr, st);
    }
    // compile keeps only KV: the last layer's attention and MLP feed nothing stored
    if (b.compile && l == c.n_layers - 1) break;
    aa.k_layer = s->k_layer(l);
    aa.v_layer = s->v_layer(l);
    if (att_tc) {
      aa.vmap = s->v_maps[2 * l];
      aa.vmap1 = s->v_maps[2 * l + 1];
      aa.sync_base = s->att_sync_total;
    }
    {
      Rec r(s, st, PIC_PROF_ATTENTION, att_bytes + (att_tc ? rot_bytes : 0), att_flops, att_launches);
      launch_attention(aa, st);
    }
    if (att_tc) {
      // the CTAs of this launch arrive at the grid-barrier counter once each
      PIC_CUDA(cudaPeekAtLastError());
      s->att_sync_total += (unsigned long long)attention_tc_grid((int)items.size());
    }
    if ((e = run_gemm(s->m->wo[l], pk(s->m->po, l), s->attn, s->h, d, H * D, T, false)) != PIC_OK) return e;
    {
      Rec r(s, st, PIC_PROF_ROWWISE, dT * dd * (4 + es), 0, 1);
      launch_rmsnorm_rows(dt, T, d, s->h, s->m->mlp_norm[l], c.rms_eps, s->x, false, nullptr, nullptr, nullptr,
                          nullptr, st);
    }
    if ((e = run_gemm(s->m->wgu[l], pk(s->m->pgu, l), s->x, s->gu_acc, 2 * F, d, T, true, PIC_PROF_GEMM_GATE_UP)) != PIC_OK)
      return e;
    {
      Rec r(s, st, PIC_PROF_ROWWISE, dT * 2 * dF * 4 + dT * dF * es, 0, 1);
      launch_swiglu(dt, T, F, s->gu_acc, s->act, st);
    }
    if ((e = run_gemm(s->m->wdown[l], pk(s->m->pdown, l), s->act, s->h, d, F, T, false)) != PIC_OK) return e;
    const bool last = l == c.n_layers - 1;
    {
      Rec r(s, st, PIC_PROF_ROWWISE, dT * dd * (4 + es), 0, 1);
      launch_rmsnorm_rows(dt, T, d, s->h, last ? s->m->final_norm : s->m->attn_norm[l + 1], c.rms_eps, s->x, last,
                          d_out, hidden_out, d_lg, s->lm_x, st);
    }
  }
  if (!b.compile && b.n_lg > 0) {
    pic_status e;
    if ((e = run_gemm(s->m->lm_head, s->m->plm, s->lm_x, logits_out, c.vocab, d, b.n_lg, true)) != PIC_OK) return e;
  }
  PIC_CUDA(cudaGetLastError());
  return PIC_OK;
}

pic_status run_forward(pic_store* s, const Batch& b, float* hidden_out, float* logits_out, cudaStream_t st) {
  // every GEMM result the forward reads is written fresh by that forward, so a forward stopped
  // part-way leaves nothing a later one depends on
  return run_forward_impl(s, b, hidden_out, logits_out, st);
}

bool valid_tokens(const int32_t* t, int n, int vocab) {
  for (int i = 0; i < n; ++i)
    if (t[i] < 0 || t[i] >= vocab) return false;
  return true;
}

// Per request, per chunk: the chunk-local indices of the tokens a link recomputes, ascending.
using Selection = std::vector<std::vector<int32_t>>;

// Handles alive, tokens in range, linked lengths within max_positions.
pic_status check_link_requests(pic_store* s, const pic_link_request* reqs, int32_t n_reqs) {
  const auto& c = s->m->cfg;
  if (n_reqs > s->cfg.max_requests) return fail(PIC_ERR_CAPACITY, "requests exceed max_requests");
  for (int r = 0; r < n_reqs; ++r) {
    const auto& q = reqs[r];
    if (q.n_chunks < 0 || (q.n_chunks > 0 && !q.chunks) || q.query_len < 1 || !q.query)
      return fail(PIC_ERR_INVALID_ARG, "invalid request");
    if (!valid_tokens(q.query, q.query_len, c.vocab)) return fail(PIC_ERR_INVALID_ARG, "query token out of range");
    long long len = q.query_len;
    for (int i = 0; i < q.n_chunks; ++i) {
      const Chunk* ch = s->live_chunk(q.chunks[i]);
      if (!ch) return fail(PIC_ERR_INVALID_ARG, "unknown chunk handle");
      len += (long long)ch->tokens.size();
    }
    if (len > s->cfg.max_positions) return fail(PIC_ERR_CAPACITY, "linked sequence exceeds max_positions");
  }
  return PIC_OK;
}

// The link proper (requests already checked): per request, in order, each chunk takes one new
// block per block holding a recomputed token (copies of those shared blocks, in ascending
// block order, lowest free ids first), then the query blocks; the recomputed rows and the
// query run through every layer, writing their K/V into those blocks.
pic_status link_selected(pic_store* s, const pic_link_request* reqs, int32_t n_reqs, const std::vector<Selection>& sels,
                         int32_t all_logits, float* hidden_out, float* logits_out, cudaStream_t st,
                         pic_request* out_requests) {
  int need = 0;
  long long rows = 0, lg_rows = 0;
  for (int r = 0; r < n_reqs; ++r) {
    for (const auto& sel : sels[r]) {
      for (size_t t = 0; t < sel.size(); ++t)
        if (!t || sel[t] / kBlock != sel[t - 1] / kBlock) ++need;
      rows += (long long)sel.size();
    }
    need += ceil_div(reqs[r].query_len, kBlock);
    rows += reqs[r].query_len;
    lg_rows += all_logits ? reqs[r].query_len : 1;
  }
  if (rows > s->cfg.max_rows) return fail(PIC_ERR_CAPACITY, "selected rows exceed max_rows");
  if (lg_rows > s->cfg.max_logit_rows) return fail(PIC_ERR_CAPACITY, "logit rows exceed max_logit_rows");
  if (!s->reserve(need)) return fail(PIC_ERR_OUT_OF_BLOCKS, "not enough free blocks for link");

  Batch b;
  std::vector<Request> made(n_reqs);
  for (int r = 0; r < n_reqs; ++r) {
    const auto& q = reqs[r];
    Request& R = made[r];
    b.begin_seq();
    int off = 0;
    for (int i = 0; i < q.n_chunks; ++i) {
      const Chunk& ch = s->chunks[q.chunks[i]];
      const std::vector<int32_t>& sel = sels[r][i];
      const int L = (int)ch.tokens.size();
      std::vector<int> mine, owner(ch.blocks.size(), -1);   // chunk blocks made private, their new copy
      for (int32_t t : sel)
        if (mine.empty() || mine.back() != t / kBlock) mine.push_back(t / kBlock);
      std::vector<int32_t> own = s->take((int)mine.size());
      for (size_t m = 0; m < mine.size(); ++m) {
        owner[mine[m]] = (int)m;
        b.copy_pairs.push_back(ch.blocks[mine[m]]);
        b.copy_pairs.push_back(own[m]);
      }
      R.private_blocks.insert(R.private_blocks.end(), own.begin(), own.end());
      for (int j = 0; j < (int)ch.blocks.size(); ++j) {
        const int blk = owner[j] >= 0 ? own[owner[j]] : ch.blocks[j];
        R.page_table.push_back(blk);
        R.page_pos.push_back(off + kBlock * j);
        R.page_len.push_back(std::min(kBlock, L - kBlock * j));
        b.page(blk, off + kBlock * j, std::min(kBlock, L - kBlock * j));
      }
      for (int32_t t : sel) {
        const int slot = own[owner[t / kBlock]] * kBlock + t % kBlock;
        R.selected.push_back(off + t);
        R.slots.push_back(slot);
        b.row(ch.tokens[t], off + t, slot);
      }
      R.chunk_ids.push_back(q.chunks[i]);
      off += L;
    }
    std::vector<int32_t> qb = s->take(ceil_div(q.query_len, kBlock));
    R.private_blocks.insert(R.private_blocks.end(), qb.begin(), qb.end());
    for (int j = 0; j < (int)qb.size(); ++j) {
      R.page_table.push_back(qb[j]);
      R.page_pos.push_back(off + kBlock * j);
      R.page_len.push_back(std::min(kBlock, q.query_len - kBlock * j));
      b.page(qb[j], off + kBlock * j, std::min(kBlock, q.query_len - kBlock * j));
    }
    for (int t = 0; t < q.query_len; ++t) {
      const int slot = qb[t / kBlock] * kBlock + t % kBlock;
      R.selected.push_back(off + t);
      R.slots.push_back(slot);
      b.row(q.query[t], off + t, slot);
      b.out_row.back() = b.n_hidden++;
      if (all_logits || t == q.query_len - 1) b.lg_row.back() = b.n_lg++;
    }
    b.end_seq();
  }
  pic_status e = run_forward(s, b, hidden_out, logits_out, st);
  if (e != PIC_OK) {
    for (auto& R : made) s->give(R.private_blocks);
    return e;
  }
  for (int r = 0; r < n_reqs; ++r) {
    for (int32_t cid : made[r].chunk_ids) s->chunks[cid].refs++;
    const int id = s->next_request++;
    s->requests[id] = std::move(made[r]);
    out_requests[r] = id;
  }
  return PIC_OK;
}

}  // namespace

extern "C" {

const char* pic_status_string(pic_status s) {
  switch (s) {
    case PIC_OK: return "PIC_OK";
    case PIC_ERR_INVALID_ARG: return "PIC_ERR_INVALID_ARG";
    case PIC_ERR_OUT_OF_BLOCKS: return "PIC_ERR_OUT_OF_BLOCKS";
    case PIC_ERR_CUDA: return "PIC_ERR_CUDA";
    case PIC_ERR_DEVICE_TIMEOUT: return "PIC_ERR_DEVICE_TIMEOUT";
    case PIC_ERR_CAPACITY: return "PIC_ERR_CAPACITY";
    case PIC_ERR_UNSUPPORTED: return "PIC_ERR_UNSUPPORTED";
    case PIC_ERR_RANGE: return "PIC_ERR_RANGE";
  }
  return "PIC_ERR_UNKNOWN";
}

const char* pic_last_error(void) { return g_last_error.c_str(); }

const char* pic_version(void) { return "pic-link 0.1 sm_103a"; }

pic_status pic_model_create(const pic_model_config* cfg, const pic_weights* w, pic_model** out) {
  if (!cfg || !w || !out) return fail(PIC_ERR_INVALID_ARG, "null argument");
  const auto& c = *cfg;
  if (c.n_layers < 1 || c.d_model < 64 || c.d_model % 64 || c.n_heads < 1 || c.n_kv_heads < 1 ||
      c.n_heads % c.n_kv_heads || (c.head_dim != 64 && c.head_dim != 128) || c.ffn_dim < 8 || c.ffn_dim % 8 ||
      c.vocab < 1 || c.block_size != kBlock || !(c.rope_base > 1.0) || !(c.rms_eps >= 0.f) ||
      (c.dtype != PIC_F32 && c.dtype != PIC_BF16) || (c.n_heads * c.head_dim) % 64)
    return fail(PIC_ERR_INVALID_ARG, "invalid model config");
  if (!w->embed || !w->lm_head || !w->final_norm || !w->attn_norm || !w->mlp_norm || !w->w_qkv || !w->w_o ||
      !w->w_gate_up || !w->w_down)
    return fail(PIC_ERR_INVALID_ARG, "null weight pointer");
  std::unique_ptr<pic_model> m(new pic_model);
  m->cfg = c;
  m->embed = w->embed;
  m->lm_head = w->lm_head;
  m->final_norm = w->final_norm;
  for (int l = 0; l < c.n_layers; ++l) {
    if (!w->attn_norm[l] || !w->mlp_norm[l] || !w->w_qkv[l] || !w->w_o[l] || !w->w_gate_up[l] || !w->w_down[l])
      return fail(PIC_ERR_INVALID_ARG, "null per-layer weight pointer");
    m->attn_norm.push_back(w->attn_norm[l]);
    m->mlp_norm.push_back(w->mlp_norm[l]);
    m->wqkv.push_back(w->w_qkv[l]);
    m->wo.push_back(w->w_o[l]);
    m->wgu.push_back(w->w_gate_up[l]);
    m->wdown.push_back(w->w_down[l]);
  }
  PIC_CUDA(cudaGetDevice(&m->device));
  PIC_CUDA(cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device));
  if (c.dtype == PIC_BF16) {
    // repack every projection matrix the tensor-core GEMM takes into contiguous 16 KB
    // tiles in their shared-memory image: each weight tile then streams from HBM as one
    // sequential bulk copy
    const int d = c.d_model, HD = c.n_heads * c.head_dim, F = c.ffn_dim, Q = m->qkv_dim();
    struct Job { const void* src; int N, K; const void** dst; };
    std::vector<Job> jobs;
    m->pqkv.assign(c.n_layers, nullptr);
    m->po.assign(c.n_layers, nullptr);
    m->pgu.assign(c.n_layers, nullptr);
    m->pdown.assign(c.n_layers, nullptr);
    for (int l = 0; l < c.n_layers; ++l) {
      jobs.push_back({m->wqkv[l], Q, d, &m->pqkv[l]});
      jobs.push_back({m->wo[l], d, HD, &m->po[l]});
      jobs.push_back({m->wgu[l], 2 * F, d, &m->pgu[l]});
      jobs.push_back({m->wdown[l], d, F, &m->pdown[l]});
    }
    jobs.push_back({m->lm_head, c.vocab, d, &m->plm});
    size_t total = 0;
    for (const Job& j : jobs)
      if (tc_gemm_supported(j.N, j.K, 1)) total += (size_t)j.N * j.K * 2;
    if (total) {
      cudaError_t e = cudaMalloc(&m->packed, total);
      if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("packed weights cudaMalloc: ") + cudaGetErrorString(e));
      size_t off = 0;
      for (const Job& j : jobs) {
        if (!tc_gemm_supported(j.N, j.K, 1)) continue;
        void* dst = (char*)m->packed + off;
        pic_status ps = tc_pack_weight(j.src, dst, j.N, j.K, 0);
        if (ps != PIC_OK) return ps;
        *j.dst = dst;
        off += (size_t)j.N * j.K * 2;
      }
      PIC_CUDA(cudaDeviceSynchronize());
      const pic_status pr = tc_check_pack_range();
      if (pr != PIC_OK) return pr;
    }
  }
  *out = m.release();
  return PIC_OK;
}

pic_status pic_model_destroy(pic_model* m) {
  delete m;
  return PIC_OK;
}

pic_status pic_store_create(pic_model* m, const pic_store_config* cfg, void* k_pool, void* v_pool, pic_store** out) {
  if (!m || !cfg || !k_pool || !v_pool || !out) return fail(PIC_ERR_INVALID_ARG, "null argument");
  const auto& sc = *cfg;
  if (sc.num_blocks < 1 || sc.max_rows < 1 || sc.max_requests < 1 || sc.max_positions < 1 || sc.max_logit_rows < 1)
    return fail(PIC_ERR_INVALID_ARG, "invalid store config");
  if (((uintptr_t)k_pool | (uintptr_t)v_pool) % 16) return fail(PIC_ERR_INVALID_ARG, "pools must be 16-byte aligned");
  const auto& c = m->cfg;
  std::unique_ptr<pic_store> s(new pic_store);
  s->m = m;
  s->cfg = sc;
  s->k_pool = k_pool;
  s->v_pool = v_pool;
  for (int32_t i = 0; i < sc.num_blocks; ++i) s->free.insert(s->free.end(), i);

  const size_t R = sc.max_rows, es = dtype_size(c.dtype);
  const size_t d = c.d_model, HD = (size_t)c.n_heads * c.head_dim, F = c.ffn_dim;
  const int rep = c.n_heads / c.n_kv_heads;
  s->att_parts_cap = 4 * m->num_sms + c.n_kv_heads * s->att_blocks_cap();
  const size_t max_pages = (size_t)sc.max_positions / kBlock + 2 * (size_t)sc.max_requests + 2;
  const size_t max_items = (size_t)s->att_parts_cap + (size_t)c.n_kv_heads * s->att_blocks_cap();
  s->meta_cap = 5 * R + 3 * max_pages * sc.max_requests + 2 * (size_t)sc.num_blocks + kAttnItemInts * max_items +
                5 * (size_t)s->att_parts_cap + 1024;

  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  const size_t as = act_size(c.dtype);
  const size_t o_h = carve(R * d * 4), o_x = carve(R * std::max(d, HD) * as),
               o_q = carve(std::max<size_t>(R, 16) * HD * 4),   // fp32 q, or >= 32 rows of fp16 q
               o_attn = carve(R * HD * as), o_act = carve(R * F * as), o_lm = carve((size_t)sc.max_logit_rows * d * as),
               o_qkv = carve(R * (size_t)m->qkv_dim() * 4), o_gu = carve(R * 2 * F * 4),
               o_atto = carve((size_t)s->att_parts_cap * kAttnPartRows * rep * c.head_dim * 4),
               o_attml = carve((size_t)s->att_parts_cap * kAttnPartRows * rep * 2 * 4), o_meta = carve(s->meta_cap * 4),
               o_rope = carve((size_t)std::max(16, sc.max_positions) * (c.head_dim / 2) * sizeof(float2));
  // ready flags of the self-zeroing GEMMs' output tiles: the most tiles any of them has
  const int rows_max = std::max(R, (size_t)sc.max_logit_rows) > 0 ? (int)std::max(R, (size_t)sc.max_logit_rows) : 1;
  // (below 1024 rows the weight tiles have 128 rows, from there 256: both row counts are covered)
  auto tiles_upto = [](int N, int T) { return std::max(tc_gemm_tiles(N, T), tc_gemm_tiles(N, std::min(T, 1023))); };
  s->tile_ready_cap = std::max({tiles_upto(std::max(128, m->qkv_dim() / 128 * 128), rows_max),
                                tiles_upto(std::max(128, 2 * c.ffn_dim / 128 * 128), rows_max),
                                tiles_upto(std::max(128, c.vocab / 128 * 128), std::max(1, sc.max_logit_rows))});
  const size_t o_ready = carve(s->tile_ready_cap * 4);
  const size_t o_sync = carve(sizeof(unsigned long long));   // the attention's grid-barrier counter
  cudaError_t e = cudaMalloc(&s->ws, off);
  if (e != cudaSuccess) return fail(PIC_ERR_CUDA, std::string("workspace cudaMalloc: ") + cudaGetErrorString(e));
  s->h = (float*)(s->ws + o_h);
  s->x = s->ws + o_x;
  s->q = (float*)(s->ws + o_q);
  s->attn = s->ws + o_attn;
  s->act = s->ws + o_act;
  s->lm_x = s->ws + o_lm;
  s->qkv_acc = (float*)(s->ws + o_qkv);
  s->gu_acc = (float*)(s->ws + o_gu);
  s->att_o = (float*)(s->ws + o_atto);
  s->att_ml = (float*)(s->ws + o_attml);
  s->meta_d = (int32_t*)(s->ws + o_meta);
  s->rope_cs = (float2*)(s->ws + o_rope);
  s->tile_ready = (int*)(s->ws + o_ready);
  s->att_sync = (unsigned long long*)(s->ws + o_sync);
  // the q rows that no forward has written yet start at zero (a 32-row box of the tensor-core
  // attention may read them), and so do the GEMMs' tile-ready flags
  e = cudaMemset(s->ws + o_q, 0, o_attn - o_q);
  if (e == cudaSuccess) e = cudaMemset(s->tile_ready, 0, s->tile_ready_cap * 4);
  if (e == cudaSuccess) e = cudaMemset(s->att_sync, 0, sizeof(unsigned long long));
  if (e != cudaSuccess) {
    cudaFree(s->ws);
    return fail(PIC_ERR_CUDA, std::string("workspace memset: ") + cudaGetErrorString(e));
  }
  e = cudaMallocHost(&s->meta_h, s->meta_cap * 4);
  if (e != cudaSuccess) {
    cudaFree(s->ws);
    return fail(PIC_ERR_CUDA, std::string("cudaMallocHost: ") + cudaGetErrorString(e));
  }
  e = cudaEventCreateWithFlags(&s->meta_ev, cudaEventDisableTiming);
  std::vector<float2> tab;
  rope_table_host(std::max(16, sc.max_positions), c.head_dim, c.rope_base, tab);
  if (e == cudaSuccess) e = cudaMemcpy(s->rope_cs, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(s->ws);
    cudaFreeHost(s->meta_h);
    return fail(PIC_ERR_CUDA, std::string("store setup: ") + cudaGetErrorString(e));
  }
  *out = s.release();
  return PIC_OK;
}

pic_status pic_store_destroy(pic_store* s) {
  if (!s) return PIC_OK;
  for (cudaEvent_t e : s->ev_pool) cudaEventDestroy(e);
  if (s->meta_ev) {
    cudaEventSynchronize(s->meta_ev);
    cudaEventDestroy(s->meta_ev);
  }
  cudaFree(s->ws);
  cudaFree(s->krot);
  cudaFree(s->sel_logits);
  cudaFreeHost(s->meta_h);
  delete s;
  return PIC_OK;
}

int32_t pic_store_free_blocks(const pic_store* s) { return s ? (int32_t)s->free.size() : -1; }

namespace {

pic_status check_compile_args(const pic_store* s, const int32_t* const* tokens, const int32_t* lens,
                              int32_t n_chunks, int32_t n_dummy, const void* out) {
  if (!s || !tokens || !lens || n_chunks < 1 || !out || n_dummy < 0 || n_dummy > kBlock)
    return fail(PIC_ERR_INVALID_ARG, "invalid compile arguments");
  for (int i = 0; i < n_chunks; ++i) {
    if (!tokens[i] || lens[i] < 1) return fail(PIC_ERR_INVALID_ARG, "empty chunk");
    if (!valid_tokens(tokens[i], lens[i], s->m->cfg.vocab)) return fail(PIC_ERR_INVALID_ARG, "token id out of range");
    if (lens[i] + n_dummy > s->cfg.max_positions) return fail(PIC_ERR_CAPACITY, "chunk longer than max_positions");
  }
  return PIC_OK;
}

// Compiles chunks `idx` of the call in one forward into newly taken blocks (evicting
// unreferenced cached chunks first if too few are free); on success out_ids[j] is the new
// chunk of idx[j] (refcount 1).
pic_status compile_batch(pic_store* s, const int32_t* const* tokens, const int32_t* lens, const std::vector<int>& idx,
                         int32_t n_dummy, cudaStream_t st, std::vector<int32_t>& out_ids) {
  long long rows = n_dummy;
  int need = 0;
  for (int i : idx) {
    rows += lens[i];
    need += ceil_div(lens[i], kBlock);
  }
  if ((int)idx.size() > s->cfg.max_requests) return fail(PIC_ERR_CAPACITY, "chunks exceed max_requests");
  if (rows > s->cfg.max_rows) return fail(PIC_ERR_CAPACITY, "compile rows exceed max_rows");
  if (!s->reserve(need)) return fail(PIC_ERR_OUT_OF_BLOCKS, "not enough free blocks for compile");
  const int n_chunks = (int)idx.size();
  Batch b;
  b.compile = true;
  // the dummy prefix is computed once per batch into the store's scratch page
  if (n_dummy > 0) {
    b.begin_seq();
    for (int j = 0; j < n_dummy; ++j) b.row(0, j, s->scratch_block() * kBlock + j);
    b.page(s->scratch_block(), 0, n_dummy);
    b.end_seq();
  }
  std::vector<std::vector<int32_t>> blocks(n_chunks);
  for (int j0 = 0; j0 < n_chunks; ++j0) {
    const int i = idx[j0];
    blocks[j0] = s->take(ceil_div(lens[i], kBlock));
    b.begin_seq();
    if (n_dummy > 0) b.page(s->scratch_block(), 0, n_dummy);
    for (int j = 0; j < (int)blocks[j0].size(); ++j)
      b.page(blocks[j0][j], n_dummy + kBlock * j, std::min(kBlock, lens[i] - kBlock * j));
    for (int t = 0; t < lens[i]; ++t)
      b.row(tokens[i][t], n_dummy + t, blocks[j0][t / kBlock] * kBlock + t % kBlock);
    b.end_seq();
  }
  pic_status e = run_forward(s, b, nullptr, nullptr, st);
  if (e != PIC_OK) {
    for (auto& bl : blocks) s->give(bl);
    return e;
  }
  out_ids.assign(n_chunks, 0);
  for (int j0 = 0; j0 < n_chunks; ++j0) {
    const int i = idx[j0];
    Chunk ch;
    ch.tokens.assign(tokens[i], tokens[i] + lens[i]);
    ch.blocks = blocks[j0];
    ch.n_dummy = n_dummy;
    const int id = s->next_chunk++;
    s->chunks[id] = std::move(ch);
    out_ids[j0] = id;
  }
  return PIC_OK;
}

}  // namespace

pic_status pic_compile(pic_store* s, const int32_t* const* tokens, const int32_t* lens, int32_t n_chunks,
                       int32_t n_dummy, pic_stream_t stream, pic_chunk* out_chunks) {
  pic_status e = check_compile_args(s, tokens, lens, n_chunks, n_dummy, out_chunks);
  if (e != PIC_OK) return e;
  std::vector<int> idx(n_chunks);
  for (int i = 0; i < n_chunks; ++i) idx[i] = i;
  std::vector<int32_t> ids;
  if ((e = compile_batch(s, tokens, lens, idx, n_dummy, (cudaStream_t)stream, ids)) != PIC_OK) return e;
  std::copy(ids.begin(), ids.end(), out_chunks);
  return PIC_OK;
}

pic_status pic_compile_cached(pic_store* s, const int32_t* const* tokens, const int32_t* lens, int32_t n_chunks,
                              int32_t n_dummy, pic_stream_t stream, pic_chunk* out_chunks, int32_t* out_hits) {
  pic_status e = check_compile_args(s, tokens, lens, n_chunks, n_dummy, out_chunks);
  if (e != PIC_OK) return e;
  // each chunk: a resident cached chunk of the same content, an earlier chunk of this call, or
  // a miss to compile
  std::vector<int32_t> hit(n_chunks, 0);
  std::vector<int> same_as(n_chunks, -1), miss;
  std::vector<uint64_t> key(n_chunks);
  for (int i = 0; i < n_chunks; ++i) {
    key[i] = content_key(tokens[i], lens[i], n_dummy);
    if ((hit[i] = s->find_cached(key[i], tokens[i], lens[i], n_dummy)) != 0) continue;
    for (int j : miss)
      if (key[j] == key[i] && lens[j] == lens[i] && std::equal(tokens[i], tokens[i] + lens[i], tokens[j])) {
        same_as[i] = j;
        break;
      }
    if (same_as[i] < 0) miss.push_back(i);
  }
  // hold the hits first so that making room for the misses cannot evict them
  for (int i = 0; i < n_chunks; ++i)
    if (hit[i]) s->ref(hit[i]);
  std::vector<int32_t> ids;
  if (!miss.empty() && (e = compile_batch(s, tokens, lens, miss, n_dummy, (cudaStream_t)stream, ids)) != PIC_OK) {
    for (int i = 0; i < n_chunks; ++i)
      if (hit[i] && --s->chunks[hit[i]].refs == 0) s->retire(hit[i]);
    return e;
  }
  std::vector<int32_t> new_id(n_chunks, 0);
  for (size_t j = 0; j < miss.size(); ++j) {
    Chunk& c = s->chunks[ids[j]];
    c.cached = true;
    c.key = key[miss[j]];
    s->cache_index.emplace(c.key, ids[j]);
    new_id[miss[j]] = ids[j];
  }
  for (int i = 0; i < n_chunks; ++i) {
    if (hit[i]) {
      out_chunks[i] = hit[i];
    } else if (same_as[i] >= 0) {
      out_chunks[i] = new_id[same_as[i]];
      s->chunks[out_chunks[i]].refs++;
    } else {
      out_chunks[i] = new_id[i];
    }
    const bool reused = hit[i] || same_as[i] >= 0;
    if (out_hits) out_hits[i] = reused ? 1 : 0;
    if (reused) ++s->cache_hits;
  }
  s->cache_misses += (int64_t)miss.size();
  return PIC_OK;
}

pic_status pic_chunk_import(pic_store* s, const int32_t* tokens, int32_t n_tokens, const void* k, const void* v,
                            pic_stream_t stream, pic_chunk* out_chunk) {
  if (!s || !tokens || n_tokens < 1 || !k || !v || !out_chunk) return fail(PIC_ERR_INVALID_ARG, "invalid import");
  const auto& c = s->m->cfg;
  if (!valid_tokens(tokens, n_tokens, c.vocab)) return fail(PIC_ERR_INVALID_ARG, "token id out of range");
  const int nb = ceil_div(n_tokens, kBlock);
  if ((size_t)nb > s->meta_cap) return fail(PIC_ERR_CAPACITY, "chunk too long for the metadata buffer");
  if (!s->reserve(nb)) return fail(PIC_ERR_OUT_OF_BLOCKS, "not enough free blocks for import");
  cudaStream_t st = (cudaStream_t)stream;
  if (s->meta_ev_pending) {
    PIC_CUDA(cudaEventSynchronize(s->meta_ev));
    s->meta_ev_pending = false;
  }
  std::vector<int32_t> blocks = s->take(nb);
  std::memcpy(s->meta_h, blocks.data(), nb * 4);
  cudaError_t e = cudaMemcpyAsync(s->meta_d, s->meta_h, nb * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaEventRecord(s->meta_ev, st);
  if (e == cudaSuccess) {
    s->meta_ev_pending = true;
    s->launches += 1;
    launch_import_kv(c.dtype, c.n_layers, n_tokens, c.n_kv_heads, c.head_dim, k, v, s->meta_d, s->blocks_total(),
                     s->k_pool, s->v_pool, st);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    s->give(blocks);
    return fail(PIC_ERR_CUDA, std::string("import: ") + cudaGetErrorString(e));
  }
  Chunk ch;
  ch.tokens.assign(tokens, tokens + n_tokens);
  ch.blocks = blocks;
  const int id = s->next_chunk++;
  s->chunks[id] = std::move(ch);
  *out_chunk = id;
  return PIC_OK;
}

pic_status pic_link(pic_store* s, const pic_link_request* reqs, int32_t n_reqs, int32_t k, int32_t all_logits,
                    float* hidden_out, float* logits_out, pic_stream_t stream, pic_request* out_requests) {
  if (!s || !reqs || n_reqs < 1 || k < 0 || !hidden_out || !logits_out || !out_requests)
    return fail(PIC_ERR_INVALID_ARG, "invalid link arguments");
  pic_status e = check_link_requests(s, reqs, n_reqs);
  if (e != PIC_OK) return e;
  // LegoLink-k: the first min(k, L) tokens of every chunk
  std::vector<Selection> sels(n_reqs);
  for (int r = 0; r < n_reqs; ++r)
    for (int i = 0; i < reqs[r].n_chunks; ++i) {
      const int L = (int)s->chunks[reqs[r].chunks[i]].tokens.size();
      std::vector<int32_t> first(std::min(k, L));
      for (int t = 0; t < (int)first.size(); ++t) first[t] = t;
      sels[r].push_back(std::move(first));
    }
  return link_selected(s, reqs, n_reqs, sels, all_logits, hidden_out, logits_out, (cudaStream_t)stream, out_requests);
}

pic_status pic_link_dynamic(pic_store* s, const pic_link_request* reqs, int32_t n_reqs, int32_t r_percent,
                            int32_t all_logits, float* hidden_out, float* logits_out, float* scores_out,
                            pic_stream_t stream, pic_request* out_requests) {
  if (!s || !reqs || n_reqs < 1 || r_percent < 0 || r_percent > 100 || !hidden_out || !logits_out || !out_requests)
    return fail(PIC_ERR_INVALID_ARG, "invalid link arguments");
  pic_status e = check_link_requests(s, reqs, n_reqs);
  if (e != PIC_OK) return e;
  const auto& c = s->m->cfg;
  const int H = c.n_heads, G = c.n_kv_heads, D = c.head_dim;
  cudaStream_t st = (cudaStream_t)stream;
  // per request: prompt length, kept count floor(r N / 100), its query rows, pages and scores
  std::vector<SelectReq> sr(n_reqs);
  std::vector<int> tok, pblk, ppos, plen;
  long long rows = 0;
  bool partial = scores_out != nullptr;
  for (int r = 0; r < n_reqs; ++r) {
    const auto& q = reqs[r];
    SelectReq& R = sr[r];
    R.row0 = (int)tok.size();
    R.lq = q.query_len;
    R.page0 = (int)pblk.size();
    R.tok0 = r ? sr[r - 1].tok0 + sr[r - 1].n_tok : 0;
    R.out0 = r ? sr[r - 1].out0 + sr[r - 1].n_pick : 0;
    R.kb0 = r ? sr[r - 1].kb0 + ceil_div(sr[r - 1].n_tok + sr[r - 1].lq, kSelectKeyBlock) : 0;
    R.pkb0 = r ? sr[r - 1].pkb0 + ceil_div(sr[r - 1].n_tok, kSelectKeyBlock) : 0;
    int N = 0;
    for (int i = 0; i < q.n_chunks; ++i) {
      const Chunk& ch = s->chunks[q.chunks[i]];
      const int L = (int)ch.tokens.size();
      for (int j = 0; j < (int)ch.blocks.size(); ++j) {
        pblk.push_back(ch.blocks[j]);
        ppos.push_back(N + kBlock * j);
        plen.push_back(std::min(kBlock, L - kBlock * j));
      }
      N += L;
    }
    R.n_tok = N;
    R.n_pages = (int)pblk.size() - R.page0;
    R.n_pick = (int)((long long)r_percent * N / 100);
    partial |= R.n_pick > 0 && R.n_pick < N;
    tok.insert(tok.end(), q.query, q.query + q.query_len);
    rows += R.n_pick + q.query_len;
  }
  if (rows > s->cfg.max_rows) return fail(PIC_ERR_CAPACITY, "selected rows exceed max_rows");
  const int n_rows = (int)tok.size();
  const int n_tok = sr.back().tok0 + sr.back().n_tok, n_out = sr.back().out0 + sr.back().n_pick;

  std::vector<Selection> sels(n_reqs);
  auto split = [&](int r, const int32_t* chosen) {   // ascending prompt positions -> per chunk
    int at = 0, off = 0;
    for (int i = 0; i < reqs[r].n_chunks; ++i) {
      const int L = (int)s->chunks[reqs[r].chunks[i]].tokens.size();
      std::vector<int32_t> mine;
      for (; at < sr[r].n_pick && chosen[at] < off + L; ++at) mine.push_back(chosen[at] - off);
      sels[r].push_back(std::move(mine));
      off += L;
    }
  };
  if (!partial) {
    // nothing or everything kept: the choice needs no scores
    for (int r = 0; r < n_reqs; ++r) {
      std::vector<int32_t> all(sr[r].n_pick);
      for (int u = 0; u < sr[r].n_pick; ++u) all[u] = u;
      split(r, all.data());
    }
  } else {
    // the scoring pass: layer-0 q, k of the query rows, then every prompt token's score
    const size_t qkv = s->m->qkv_dim();
    const size_t ml_floats = (size_t)n_rows * H * 2, sc_floats = scores_out ? 0 : (size_t)n_tok;
    if (ml_floats + sc_floats > (size_t)s->cfg.max_rows * 2 * c.ffn_dim)
      return fail(PIC_ERR_CAPACITY, "prompt tokens exceed the scoring workspace");
    // every query row's logits against every key it may see, per request
    size_t n_logits = 0;
    for (SelectReq& R : sr) {
      if (n_logits > (size_t)INT32_MAX) break;
      R.lg0 = (int)n_logits;
      n_logits += (size_t)R.lq * H * (R.n_tok + R.lq);
    }
    if (n_logits > (size_t)INT32_MAX) return fail(PIC_ERR_CAPACITY, "dynamic selection: too many query-key logits");
    if (n_logits > s->sel_logits_cap) {
      // cudaFree waits for the kernels still reading the old scratch
      PIC_CUDA(cudaFree(s->sel_logits));
      s->sel_logits = nullptr;
      s->sel_logits_cap = 0;
      PIC_CUDA(cudaMalloc(&s->sel_logits, n_logits * sizeof(float)));
      s->sel_logits_cap = n_logits;
    }
    const size_t n_int = tok.size() + 3 * pblk.size() + (size_t)kSelectReqInts * n_reqs + n_out;
    if (n_int > s->meta_cap) return fail(PIC_ERR_CAPACITY, "metadata exceeds workspace");
    if (s->meta_ev_pending) {
      PIC_CUDA(cudaEventSynchronize(s->meta_ev));
      s->meta_ev_pending = false;
    }
    int32_t* hp = s->meta_h;
    size_t o = 0;
    auto put = [&](const void* src, size_t n) {
      if (n) std::memcpy(hp + o, src, n * 4);
      const size_t at = o;
      o += n;
      return s->meta_d + at;
    };
    const int* d_tok = put(tok.data(), tok.size());
    const int* d_pblk = put(pblk.data(), pblk.size());
    const int* d_ppos = put(ppos.data(), ppos.size());
    const int* d_plen = put(plen.data(), plen.size());
    const SelectReq* d_req = (const SelectReq*)put(sr.data(), (size_t)kSelectReqInts * n_reqs);
    const size_t o_chosen = o;
    PIC_CUDA(cudaMemcpyAsync(s->meta_d, hp, o * 4, cudaMemcpyHostToDevice, st));
    const int es = (int)dtype_size(c.dtype);
    {
      Rec rc(s, st, PIC_PROF_ROWWISE, (double)n_rows * c.d_model * (es + 4 + es), 0, 1);
      launch_embed_norm(c.dtype, n_rows, c.d_model, s->m->embed, d_tok, s->m->attn_norm[0], c.rms_eps, s->h, s->x,
                        st);
    }
    {
      const bool pk = !s->m->pqkv.empty();
      const bool zero_kernel = !(pk && tc_gemm_tiles((int)qkv, n_rows) <= s->tile_ready_cap);
      Rec rc(s, st, PIC_PROF_GEMM, (double)qkv * c.d_model * es + (double)n_rows * (c.d_model * es + qkv * 8),
             2.0 * qkv * c.d_model * n_rows, 1 + (zero_kernel ? 1 : 0));
      if ((e = gemm(s, s->m->wqkv[0], pk ? s->m->pqkv[0] : nullptr, s->x, s->qkv_acc, (int)qkv, c.d_model, n_rows, st,
                    true)) != PIC_OK)
        return e;
    }
    SelectArgs a{};
    a.reqs = d_req;
    a.n_reqs = n_reqs;
    a.n_rows = n_rows;
    a.n_tok = n_tok;
    a.H = H;
    a.G = G;
    a.qkv = s->qkv_acc;
    a.k_layer0 = s->k_layer(0);
    a.page_block = d_pblk;
    a.page_pos = d_ppos;
    a.page_len = d_plen;
    a.rope_cs = s->rope_cs;
    a.qrot = s->q;
    a.logits = s->sel_logits;
    a.n_kb = sr.back().kb0 + ceil_div(sr.back().n_tok + sr.back().lq, kSelectKeyBlock);
    a.n_pkb = sr.back().pkb0 + ceil_div(sr.back().n_tok, kSelectKeyBlock);
    a.ml = s->gu_acc;
    a.scores = scores_out ? scores_out : s->gu_acc + ml_floats;
    a.chosen = s->meta_d + o_chosen;
    {
      double pairs = 0;   // (query row, visible key) pairs: one logit each
      for (const SelectReq& R : sr) pairs += (double)R.lq * R.n_tok + (double)R.lq * (R.lq + 1) / 2;
      Rec rc(s, st, PIC_PROF_SELECT, (double)n_tok * G * D * es + (double)n_rows * H * D * 8 + 3.0 * n_logits * 4,
             pairs * H * D * 2.0, 5);
      if ((e = launch_select(a, D, c.dtype, st)) != PIC_OK) return e;
    }
    if (n_out) PIC_CUDA(cudaMemcpyAsync(hp + o_chosen, a.chosen, (size_t)n_out * 4, cudaMemcpyDeviceToHost, st));
    PIC_CUDA(cudaStreamSynchronize(st));
    for (int r = 0; r < n_reqs; ++r) {
      const int32_t* ch = hp + o_chosen + sr[r].out0;
      for (int i = 0; i < sr[r].n_pick; ++i)
        if (ch[i] < 0 || ch[i] >= sr[r].n_tok || (i && ch[i] <= ch[i - 1]))
          return fail(PIC_ERR_CUDA, "token selection returned an invalid position list");
      split(r, ch);
    }
  }
  return link_selected(s, reqs, n_reqs, sels, all_logits, hidden_out, logits_out, st, out_requests);
}

pic_status pic_decode(pic_store* s, const pic_request* reqs, const int32_t* tokens, int32_t n_reqs,
                      float* hidden_out, float* logits_out, pic_stream_t stream, int32_t* out_positions,
                      int32_t* out_slots) {
  if (!s || !reqs || !tokens || n_reqs < 1 || !hidden_out || !logits_out)
    return fail(PIC_ERR_INVALID_ARG, "invalid decode arguments");
  const auto& c = s->m->cfg;
  if (n_reqs > s->cfg.max_requests) return fail(PIC_ERR_CAPACITY, "requests exceed max_requests");
  if (n_reqs > s->cfg.max_rows) return fail(PIC_ERR_CAPACITY, "decode rows exceed max_rows");
  if (n_reqs > s->cfg.max_logit_rows) return fail(PIC_ERR_CAPACITY, "logit rows exceed max_logit_rows");
  if (!valid_tokens(tokens, n_reqs, c.vocab)) return fail(PIC_ERR_INVALID_ARG, "token id out of range");
  // validate and count new blocks (nothing is allocated before every check passes)
  std::set<int32_t> seen;
  int need = 0;
  for (int i = 0; i < n_reqs; ++i) {
    auto it = s->requests.find(reqs[i]);
    if (it == s->requests.end()) return fail(PIC_ERR_INVALID_ARG, "unknown request handle");
    if (!seen.insert(reqs[i]).second) return fail(PIC_ERR_INVALID_ARG, "a request appears twice in one decode");
    const Request& R = it->second;
    if (R.page_pos.back() + R.page_len.back() >= s->cfg.max_positions)
      return fail(PIC_ERR_CAPACITY, "decoded sequence exceeds max_positions");
    if (R.page_len.back() == kBlock) ++need;
  }
  if (!s->reserve(need)) return fail(PIC_ERR_OUT_OF_BLOCKS, "not enough free blocks for decode");

  // one sequence per request: its whole page table, the last page one row longer (or a new
  // page), and the new row at the next position
  Batch b;
  std::vector<int32_t> fresh(n_reqs, -1), pos(n_reqs), slot(n_reqs);
  for (int i = 0; i < n_reqs; ++i) {
    const Request& R = s->requests[reqs[i]];
    const int np = (int)R.page_table.size(), last_len = R.page_len.back();
    pos[i] = R.page_pos.back() + last_len;
    b.begin_seq();
    for (int j = 0; j < np; ++j)
      b.page(R.page_table[j], R.page_pos[j], R.page_len[j] + (j == np - 1 && last_len < kBlock ? 1 : 0));
    if (last_len == kBlock) {
      fresh[i] = s->take(1)[0];
      b.page(fresh[i], pos[i], 1);
      slot[i] = fresh[i] * kBlock;
    } else {
      slot[i] = R.page_table.back() * kBlock + last_len;
    }
    b.row(tokens[i], pos[i], slot[i]);
    b.out_row.back() = b.n_hidden++;
    b.lg_row.back() = b.n_lg++;
    b.end_seq();
  }
  pic_status e = run_forward(s, b, hidden_out, logits_out, (cudaStream_t)stream);
  if (e != PIC_OK) {
    for (int32_t f : fresh)
      if (f >= 0) s->give({f});
    return e;
  }
  for (int i = 0; i < n_reqs; ++i) {
    Request& R = s->requests[reqs[i]];
    if (fresh[i] >= 0) {
      R.page_table.push_back(fresh[i]);
      R.page_pos.push_back(pos[i]);
      R.page_len.push_back(1);
      R.private_blocks.push_back(fresh[i]);
    } else {
      R.page_len.back() += 1;
    }
    if (out_positions) out_positions[i] = pos[i];
    if (out_slots) out_slots[i] = slot[i];
  }
  return PIC_OK;
}

pic_status pic_request_get_info(const pic_store* s, pic_request r, pic_request_info* out) {
  if (!s || !out) return fail(PIC_ERR_INVALID_ARG, "null argument");
  auto it = s->requests.find(r);
  if (it == s->requests.end()) return fail(PIC_ERR_INVALID_ARG, "unknown request handle");
  const Request& R = it->second;
  out->n_selected = (int32_t)R.selected.size();
  out->selected = R.selected.data();
  out->slots = R.slots.data();
  out->n_pages = (int32_t)R.page_table.size();
  out->page_table = R.page_table.data();
  out->page_pos = R.page_pos.data();
  out->page_len = R.page_len.data();
  out->n_private = (int32_t)R.private_blocks.size();
  out->private_blocks = R.private_blocks.data();
  return PIC_OK;
}

pic_status pic_chunk_get_blocks(const pic_store* s, pic_chunk c, int32_t* n_blocks, const int32_t** blocks) {
  if (!s || !n_blocks || !blocks) return fail(PIC_ERR_INVALID_ARG, "null argument");
  auto it = s->chunks.find(c);
  if (it == s->chunks.end() || it->second.refs < 1) return fail(PIC_ERR_INVALID_ARG, "unknown chunk handle");
  *n_blocks = (int32_t)it->second.blocks.size();
  *blocks = it->second.blocks.data();
  return PIC_OK;
}

pic_status pic_release_chunk(pic_store* s, pic_chunk c) {
  if (!s) return fail(PIC_ERR_INVALID_ARG, "null store");
  Chunk* ch = s->live_chunk(c);
  if (!ch) return fail(PIC_ERR_INVALID_ARG, "unknown chunk handle");
  if (--ch->refs == 0) s->retire(c);
  return PIC_OK;
}

pic_status pic_release_request(pic_store* s, pic_request r) {
  if (!s) return fail(PIC_ERR_INVALID_ARG, "null store");
  auto it = s->requests.find(r);
  if (it == s->requests.end()) return fail(PIC_ERR_INVALID_ARG, "unknown request handle");
  s->give(it->second.private_blocks);
  for (int32_t cid : it->second.chunk_ids) {
    auto ci = s->chunks.find(cid);
    if (ci != s->chunks.end() && ci->second.refs > 0 && --ci->second.refs == 0) s->retire(cid);
  }
  s->requests.erase(it);
  return PIC_OK;
}

pic_status pic_store_get_cache_stats(const pic_store* s, pic_cache_stats* out) {
  if (!s || !out) return fail(PIC_ERR_INVALID_ARG, "null argument");
  std::memset(out, 0, sizeof(*out));
  out->hits = s->cache_hits;
  out->misses = s->cache_misses;
  out->evictions = s->cache_evictions;
  for (const auto& kv : s->chunks)
    if (kv.second.cached) {
      ++out->cached_chunks;
      if (kv.second.refs == 0) {
        ++out->unreferenced_chunks;
        out->unreferenced_blocks += (int32_t)kv.second.blocks.size();
      }
    }
  out->blocks_in_use = s->cfg.num_blocks - (int32_t)s->free.size();
  out->block_bytes = (int64_t)s->block_bytes() * 2 * s->m->cfg.n_layers;
  return PIC_OK;
}

pic_status pic_store_evict(pic_store* s, int32_t max_chunks, int32_t* n_evicted) {
  if (!s) return fail(PIC_ERR_INVALID_ARG, "null store");
  int32_t n = 0;
  while (!s->lru.empty() && (max_chunks < 0 || n < max_chunks)) {
    s->evict_front();
    ++n;
  }
  if (n_evicted) *n_evicted = n;
  return PIC_OK;
}

pic_status pic_profile_begin(pic_store* s) {
  if (!s) return fail(PIC_ERR_INVALID_ARG, "null store");
  s->prof.clear();
  s->ev_used = 0;
  s->prof_on = true;
  return PIC_OK;
}

pic_status pic_profile_end(pic_store* s, pic_profile* out) {
  if (!s || !out) return fail(PIC_ERR_INVALID_ARG, "null argument");
  std::memset(out, 0, sizeof(*out));
  s->prof_on = false;
  for (const auto& r : s->prof) {
    PIC_CUDA(cudaEventSynchronize(r.b));
    float ms = 0.f;
    PIC_CUDA(cudaEventElapsedTime(&ms, r.a, r.b));
    out->launches[r.cls] += r.launches;
    out->ms[r.cls] += ms;
    out->bytes[r.cls] += r.bytes;
    out->flops[r.cls] += r.flops;
  }
  out->total_launches = s->launches;
  s->prof.clear();
  s->ev_used = 0;
  return PIC_OK;
}

int64_t pic_store_launch_count(const pic_store* s) { return s ? s->launches : -1; }

pic_status pic_sync(pic_store* s, pic_stream_t stream) {
  (void)s;
  PIC_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  // every flag is read (and cleared) even when an earlier one is set
  const pic_status a = attn_check_timeout();
  const pic_status g = tc_check_timeout();
  const pic_status r = rows_check_range();
  return a != PIC_OK ? a : g != PIC_OK ? g : r;
}

pic_status pic_debug_raise_device_flag(int32_t which) {
  switch (which) {
    case 1: attn_raise_timeout(); break;
    case 2: tc_raise_timeout(); break;
    case 3: rows_raise_range(); break;
    default: return fail(PIC_ERR_INVALID_ARG, "device flag must be 1, 2 or 3");
  }
  PIC_CUDA(cudaGetLastError());
  return PIC_OK;
}

}  // extern "C"
