/*
 * pic.h — C ABI of the position-independent KV link library (GB300, sm_103a).
 *
 * The library implements position-independent context caching (PIC) as two steps:
 *
 *   compile  prefill one immutable chunk on its own, with position ids starting at 0,
 *            and store its per-layer K (before RoPE) and V in 16-token pages.
 *            ("EPIC: Efficient Position-Independent Caching for Serving Large Language
 *            Models", summary page, Approach.)
 *   link     LegoLink-k: for a prompt made of compiled chunks plus a query suffix,
 *            recompute only the first k tokens of every chunk and all query tokens,
 *            through every layer, attending causally to the reused KV of every
 *            earlier chunk; RoPE is applied to each key at attention time from its
 *            absolute position. Each chunk's first ceil(k/16) pages become
 *            request-private copies; every other page stays shared.
 *            (EPIC summary page, Approach; "MEPIC: Memory Efficient Position
 *            Independent Caching for LLM Serving", abstract.)
 *
 * Conventions
 *   - Every call returns pic_status; nothing throws or aborts across the ABI.
 *     pic_last_error() gives a message for the last failure on the calling thread.
 *   - A failing call leaves no partial state: block allocation is all-or-nothing.
 *   - Device pointers passed in (weights, KV pools, outputs) are BORROWED: the caller
 *     allocates them, keeps them alive while the model/store uses them, and frees them.
 *     Handles (pic_model*, pic_store*, pic_chunk, pic_request) are OWNED by the library
 *     and freed by the matching destroy/release call.
 *   - GPU work is asynchronous on the caller's stream (cudaStream_t; NULL = legacy
 *     default stream). Host-side metadata outputs are valid when the call returns.
 *     Device-side wait timeouts are reported by pic_sync().
 *   - Handles are not thread-safe: one thread at a time per store.
 *   - Block size is 16 tokens. KV pool layout (per pool, K and V alike):
 *       [n_layers][num_blocks + 1][n_kv_heads][16][head_dim] in the model dtype.
 *     Block index num_blocks is the store's own scratch page (dummy-prefix rows
 *     during a LegoLink-0 compile); ids 0..num_blocks-1 are allocated to chunks and
 *     requests. K is stored without positional encoding.
 */
#ifndef PIC_H_
#define PIC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pic_stream_t; /* identical to cudaStream_t */

typedef enum {
  PIC_OK = 0,
  PIC_ERR_INVALID_ARG = 1,     /* bad size, pointer, handle or layout */
  PIC_ERR_OUT_OF_BLOCKS = 2,   /* the pool cannot hold the new blocks; nothing changed */
  PIC_ERR_CUDA = 3,            /* a CUDA runtime call failed (message in pic_last_error) */
  PIC_ERR_DEVICE_TIMEOUT = 4,  /* a kernel gave up a bounded wait; its outputs are invalid */
  PIC_ERR_CAPACITY = 5,        /* the call exceeds a capacity fixed at store creation */
  PIC_ERR_UNSUPPORTED = 6,     /* shape/dtype combination not built */
  PIC_ERR_RANGE = 7            /* a value bound for an fp16 tensor-core operand was outside fp16's
                                  range; the outputs since the last pic_sync are invalid */
} pic_status;

typedef enum { PIC_F32 = 0, PIC_BF16 = 1 } pic_dtype;

typedef int32_t pic_chunk;    /* > 0 when valid */
typedef int32_t pic_request;  /* > 0 when valid */

/* Llama-style pre-norm decoder: RMSNorm, rotate-half RoPE (theta_i = base^(-2i/D)),
 * GQA (query head h reads KV head h / (n_heads / n_kv_heads)), SwiGLU MLP, final
 * RMSNorm, untied LM head, no biases. */
typedef struct {
  int32_t n_layers;
  int32_t d_model;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t head_dim;   /* 64 or 128 */
  int32_t ffn_dim;
  int32_t vocab;
  double rope_base;
  float rms_eps;
  int32_t dtype;      /* pic_dtype of weights, KV pools and GEMM operands; accumulation is fp32 */
  int32_t block_size; /* must be 16 */
} pic_model_config;

/* Device pointers (borrowed). Matrices are row-major [out][in] (nn.Linear layout) in
 * the model dtype; norm gains are fp32. The per-layer arrays are HOST arrays of
 * n_layers device pointers; the library copies the arrays at model creation. */
typedef struct {
  const void* embed;              /* [vocab][d_model] */
  const void* lm_head;            /* [vocab][d_model] */
  const float* final_norm;        /* [d_model] */
  const float* const* attn_norm;  /* per layer [d_model] */
  const float* const* mlp_norm;   /* per layer [d_model] */
  const void* const* w_qkv;       /* per layer [(n_heads + 2 n_kv_heads) head_dim][d_model]: Q rows, K rows, V rows */
  const void* const* w_o;         /* per layer [d_model][n_heads head_dim] */
  const void* const* w_gate_up;   /* per layer [2 ffn_dim][d_model]: gate rows, then up rows */
  const void* const* w_down;      /* per layer [d_model][ffn_dim] */
} pic_weights;

typedef struct pic_model pic_model;
typedef struct pic_store pic_store;

/* Capacities fixed at store creation (they size the library-owned device workspace). */
typedef struct {
  int32_t num_blocks;        /* allocatable pages; pools hold num_blocks + 1 */
  int32_t max_rows;          /* rows computed by one compile or link call (all requests) */
  int32_t max_requests;      /* requests (or chunks) in one call */
  int32_t max_positions;     /* longest linked sequence, in tokens */
  int32_t max_logit_rows;    /* rows of logits one link may produce */
} pic_store_config;

/* One request of a link batch. `chunks` and `query` are host arrays. */
typedef struct {
  const pic_chunk* chunks;   /* compiled chunks in prompt order (repeats allowed) */
  int32_t n_chunks;
  const int32_t* query;      /* query-suffix token ids */
  int32_t query_len;         /* >= 1 */
} pic_link_request;

/* Host metadata of a linked request; arrays are owned by the store and stay valid
 * until the request is released. All int32. */
typedef struct {
  int32_t n_selected;
  const int32_t* selected;        /* absolute positions of recomputed rows, ascending */
  const int32_t* slots;           /* block_id * 16 + row of each selected row */
  int32_t n_pages;
  const int32_t* page_table;      /* physical block of each page, in position order */
  const int32_t* page_pos;        /* absolute position of row 0 of each page */
  const int32_t* page_len;        /* valid rows of each page (ragged chunk tails) */
  int32_t n_private;
  const int32_t* private_blocks;  /* blocks owned by this request (chunk privates, then query) */
} pic_request_info;

const char* pic_status_string(pic_status s);
const char* pic_last_error(void);
/* Library version string and the CUDA arch it was built for ("sm_103a"). */
const char* pic_version(void);

/* Creates a model on the current CUDA device. Validates the config (head_dim 64/128,
 * n_heads % n_kv_heads == 0, d_model % 64 == 0, dims multiples of 8) and, for bf16,
 * repacks the bf16 projection matrices into a library-owned tensor-core tile copy
 * (pic_op_pack_weight layout; the originals stay borrowed and are still read for the
 * embedding gather). */
pic_status pic_model_create(const pic_model_config* cfg, const pic_weights* w, pic_model** out);
pic_status pic_model_destroy(pic_model* m);

/* Creates a paged store over caller-owned K/V pools (layout in the header comment).
 * Allocates the library-owned device workspace and the RoPE table (fp64 angles on
 * the host, stored fp32). bf16 models with head_dim 128 and 4 query heads per KV head
 * (the tensor-core attention) also use a device scratch holding one layer's K of every
 * page of a forward, rotated to each row's position (fp16, 4 KB per page and KV head):
 * the store allocates it at the first compile, link or decode that needs it and grows it
 * (a cudaFree + cudaMalloc, which synchronizes the device) when a later call has more
 * pages; it is freed with the store. */
pic_status pic_store_create(pic_model* m, const pic_store_config* cfg, void* k_pool, void* v_pool,
                            pic_store** out);
pic_status pic_store_destroy(pic_store* s);
int32_t pic_store_free_blocks(const pic_store* s);

/* compile: prefill `n_chunks` chunks independently (each from position 0, behind
 * n_dummy dummy tokens of id 0 whose KV is then discarded; n_dummy in 0..16) and store
 * each in ceil(L/16) blocks, lowest free ids first, in chunk order. tokens[i] are host
 * arrays of lens[i] >= 1 ids. Each new chunk has refcount 1. */
pic_status pic_compile(pic_store* s, const int32_t* const* tokens, const int32_t* lens, int32_t n_chunks,
                       int32_t n_dummy, pic_stream_t stream, pic_chunk* out_chunks);

/* Stores externally produced chunk KV as if compiled: k, v are DEVICE arrays
 * [n_layers][n_tokens][n_kv_heads][head_dim] (pre-RoPE K) in the model dtype, copied
 * into ceil(n_tokens/16) new blocks. tokens (host) are kept for link recomputation. */
pic_status pic_chunk_import(pic_store* s, const int32_t* tokens, int32_t n_tokens, const void* k, const void* v,
                            pic_stream_t stream, pic_chunk* out_chunk);

/* link (LegoLink-k) over a batch of requests. Per request, in order: each chunk gets
 * ceil(min(k, L_i)/16) private blocks (copies of its first shared blocks), then
 * ceil(query_len/16) query blocks. Selected rows = first min(k, L_i) rows of every
 * chunk + all query rows, at contiguous absolute positions. Recomputed pre-RoPE K/V
 * are written into the private/query blocks of every layer.
 * Outputs (device, caller-owned, fp32):
 *   hidden_out [sum query_len][d_model]  final-normed hidden of every query row;
 *   logits_out [n_reqs][vocab] (last query row per request), or
 *              [sum query_len][vocab] when all_logits != 0.
 * out_requests (host, n_reqs) receives the request handles. */
pic_status pic_link(pic_store* s, const pic_link_request* reqs, int32_t n_reqs, int32_t k, int32_t all_logits,
                    float* hidden_out, float* logits_out, pic_stream_t stream, pic_request* out_requests);

/* link with dynamic (attention-based) token selection -- the CacheBlend-r step the EPIC pages
 * compare LegoLink's static choice against (EPIC summary page: problem statement; Measured
 * effects table, CacheBlend-r rows and the static-vs-dynamic row). Per request, with N prompt
 * tokens (the chunks' total length) and query_len query tokens:
 *   1. score: the query rows' layer-0 q and k are computed (embedding, RMSNorm, QKV
 *      projection); each query row and head attends causally, RoPE at absolute positions,
 *      over the prompt's compiled layer-0 K (nothing recomputed) and the query's own k; a
 *      prompt token's score is the sum of the softmax weights it receives over all query rows
 *      and heads (fp32);
 *   2. choose: the floor(r_percent * N / 100) tokens with the largest scores, equal scores
 *      taken in ascending position order;
 *   3. link: as pic_link, with the chosen tokens in place of each chunk's first k: every
 *      chunk block holding a chosen token becomes a private copy (per request, per chunk in
 *      order, ascending block order, lowest free ids first), then the query blocks; the
 *      chosen rows and the query run through every layer.
 * r_percent = 0 recomputes only the query (naive reuse); r_percent = 100 recomputes every
 * token (full recompute). The chosen positions are the request's selected list
 * (pic_request_get_info), followed by the query positions. Steps 1-2 run on the stream and
 * the call waits for them (the plan of step 3 needs the choice); step 3 is asynchronous as
 * in pic_link. Scoring is skipped when the choice does not depend on it (every request keeps
 * none or all of its tokens) and scores_out is NULL.
 * scores_out: NULL, or a device fp32 array of sum(N) that receives every request's token
 * scores in order. Capacities as pic_link (sum of kept tokens + query rows <= max_rows);
 * PIC_ERR_CAPACITY also when the scoring scratch (2 x query rows x n_heads + sum(N) floats,
 * the latter only when scores_out is NULL) exceeds max_rows x 2 x ffn_dim floats, or when
 * the pass's logits (query_len x n_heads x (N + query_len) per request) exceed 2^31 floats.
 * The logits live in a device scratch the store allocates at the first scoring pass and grows
 * (cudaFree + cudaMalloc, which synchronize the device) when a later pass needs more; it is
 * freed with the store. */
pic_status pic_link_dynamic(pic_store* s, const pic_link_request* reqs, int32_t n_reqs, int32_t r_percent,
                            int32_t all_logits, float* hidden_out, float* logits_out, float* scores_out,
                            pic_stream_t stream, pic_request* out_requests);

/* decode: one generated token per linked request, after its link -- the step that turns the
 * linked prompt into output tokens (time to first token ends at the link's logits; EPIC
 * summary page, Measured effects table). For each i, host token tokens[i] is appended to
 * request reqs[i] at the position after the request's last one (its last query row or last
 * decoded token) and runs through every layer: its pre-RoPE K and V go into the next row of
 * the request's last page, or, when that page is full, into row 0 of a new block (lowest
 * free id, requests in call order; the block joins the request's private blocks and page
 * table); its query attends causally to every row of the request's pages -- the reused and
 * recomputed chunk rows, the query rows, earlier decoded rows -- and to itself, with RoPE
 * applied inside the attention at each key's absolute position, as in link.
 * Requests must be distinct and alive. n_reqs <= max_requests, max_rows and max_logit_rows;
 * each request's new length <= max_positions (else PIC_ERR_CAPACITY). PIC_ERR_OUT_OF_BLOCKS
 * when the pool cannot give every request that needs one a new block; then nothing changes.
 * Outputs (device, caller-owned, fp32): hidden_out [n_reqs][d_model] final-normed hidden of
 * each new row; logits_out [n_reqs][vocab]. out_positions, out_slots (host int32 [n_reqs],
 * either may be NULL): the new rows' absolute positions and slots (block_id * 16 + row).
 * pic_request_get_info reports the grown page table afterwards; its selected/slots lists
 * stay those of the link. */
pic_status pic_decode(pic_store* s, const pic_request* reqs, const int32_t* tokens, int32_t n_reqs,
                      float* hidden_out, float* logits_out, pic_stream_t stream, int32_t* out_positions,
                      int32_t* out_slots);

pic_status pic_request_get_info(const pic_store* s, pic_request r, pic_request_info* out);

/* compile with content-addressed reuse. PIC compiles each chunk once and links it into any
 * prompt (EPIC summary page, Approach); MEPIC keeps one shared copy of a chunk's KV in HBM for
 * every request that uses it (abstract). For each chunk, a resident chunk that an earlier
 * pic_compile_cached made from the same tokens and n_dummy is returned instead of compiling
 * again (one more
 * reference; out_hits[i] = 1), and identical chunks within the call are compiled once; the
 * others are compiled in one batch, as pic_compile does (out_hits[i] = 0). out_hits (host
 * [n_chunks]) may be NULL. Chunks made by this call are "cached": when their last reference
 * (handles and requests) is released they stay resident, their handles no longer valid,
 * until reused by a later pic_compile_cached or evicted. Every call that needs blocks
 * (compile, import, link, decode) and finds too few free ones first evicts unreferenced
 * cached chunks, least recently released first -- only if that frees enough; otherwise it
 * fails with PIC_ERR_OUT_OF_BLOCKS and evicts nothing. Evictions are not undone if the call
 * then fails for another reason. Chunks from pic_compile and pic_chunk_import are never
 * cached: their blocks return to the pool at their last release, as before. */
pic_status pic_compile_cached(pic_store* s, const int32_t* const* tokens, const int32_t* lens, int32_t n_chunks,
                              int32_t n_dummy, pic_stream_t stream, pic_chunk* out_chunks, int32_t* out_hits);

/* Counters of the content-addressed reuse and the pool's occupancy (HBM in use by KV pages =
 * blocks_in_use x block_bytes). */
typedef struct {
  int64_t hits;                 /* pic_compile_cached chunks served without compiling */
  int64_t misses;               /* chunks it compiled */
  int64_t evictions;            /* unreferenced cached chunks evicted to free blocks */
  int32_t cached_chunks;        /* resident cached chunks, referenced or not */
  int32_t unreferenced_chunks;  /* of those, the evictable ones */
  int32_t unreferenced_blocks;  /* blocks held by the evictable ones */
  int32_t blocks_in_use;        /* allocated blocks: num_blocks - free */
  int64_t block_bytes;          /* bytes of one block id in both pools over all layers */
} pic_cache_stats;
pic_status pic_store_get_cache_stats(const pic_store* s, pic_cache_stats* out);
/* Evicts up to max_chunks (all when < 0) unreferenced cached chunks, least recently released
 * first; n_evicted (may be NULL) receives the count. */
pic_status pic_store_evict(pic_store* s, int32_t max_chunks, int32_t* n_evicted);
/* Blocks of a chunk (owned by the store, valid while the chunk lives). */
pic_status pic_chunk_get_blocks(const pic_store* s, pic_chunk c, int32_t* n_blocks, const int32_t** blocks);

/* Drops the caller's reference; blocks return to the pool when no request uses the chunk. */
pic_status pic_release_chunk(pic_store* s, pic_chunk c);
/* Frees the request's private and query blocks and drops its chunk references. */
pic_status pic_release_request(pic_store* s, pic_request r);

/* Waits for the stream and reports what the kernels flagged since the last pic_sync (the
 * flags are then cleared): PIC_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait, else
 * PIC_ERR_RANGE if a value bound for an fp16 tensor-core operand of a bf16 model was outside
 * fp16's finite range or NaN -- a normed or SwiGLU activation or a rotated, scaled q above
 * 65504 in magnitude, a stored V above 65504 or a stored K above 46000 (RoPE can grow a K
 * component by up to sqrt 2). The pages fix no precision beyond bf16 storage; the fp16
 * operands are this library's reading, and this check is where a model outside it shows.
 * s may be NULL. */
pic_status pic_sync(pic_store* s, pic_stream_t stream);

/* Sets one of the device flags that pic_sync reports, from the host, without running a
 * kernel: 1 = the tensor-core attention's bounded-wait timeout, 2 = the tensor-core GEMM's,
 * 3 = the fp16 range flag. Lets a caller (and the tests) exercise its handling of those
 * statuses without making a kernel wait or overflow. PIC_ERR_INVALID_ARG for other values. */
pic_status pic_debug_raise_device_flag(int32_t which);

/* ------------------------------------------------------------------ profiling
 * Between pic_profile_begin and pic_profile_end the store brackets each of its kernel
 * launches with CUDA events on the launch stream and records the algorithmic bytes and
 * FLOPs of that launch (operands read once, results written once). Launch counting is
 * always on. Classes: */
enum {
  PIC_PROF_GEMM = 0,       /* tcgen05 / SIMT projection GEMMs (incl. LM head) except gate/up */
  PIC_PROF_ATTENTION = 1,  /* paged attention + split merge */
  PIC_PROF_ROWWISE = 2,    /* embedding/norm, split-K epilogues, SwiGLU */
  PIC_PROF_COPY = 3,       /* request-private block copies, KV import, accumulator zeroing */
  PIC_PROF_GEMM_GATE_UP = 4, /* the MLP gate/up projection GEMM (the largest weight stream) */
  PIC_PROF_SELECT = 5,     /* dynamic selection: token scoring and top-r choice */
  PIC_PROF_CLASSES = 6
};
typedef struct {
  int64_t launches[PIC_PROF_CLASSES];  /* kernel launches recorded while profiling */
  double ms[PIC_PROF_CLASSES];         /* summed event time of those launches */
  double bytes[PIC_PROF_CLASSES];      /* summed algorithmic bytes */
  double flops[PIC_PROF_CLASSES];      /* summed algorithmic FLOPs */
  int64_t total_launches;              /* all kernel launches by this store since creation */
} pic_profile;

pic_status pic_profile_begin(pic_store* s);
/* Synchronizes the recorded streams, fills `out` and stops recording. */
pic_status pic_profile_end(pic_store* s, pic_profile* out);
/* Kernel launches made by this store since creation (host counter, no sync). */
int64_t pic_store_launch_count(const pic_store* s);

/* ------------------------------------------------------------------ kernel-level calls
 * Single steps of the link path, exposed for testing and profiling. All pointers are
 * device pointers unless stated; all work is async on `stream`.
 */

/* Y[T][N] (fp32, overwritten) = X[T][K] . W[N][K]^T, both operands in `dtype`.
 * bf16 runs on the tcgen05 tensor-core kernel when K % 64 == 0 and N % 128 == 0 (rows
 * 16-byte aligned; split-K partial sums meet in Y through TMA bulk reduce-adds), fp32 and
 * other shapes on the SIMT kernel. Needs no scratch. */
pic_status pic_op_gemm(int32_t dtype, const void* W, const void* X, float* Y, int32_t N, int32_t K, int32_t T,
                       pic_stream_t stream);

/* Repacks a bf16 [N][K] matrix (N % 128 == 0, K % 64 == 0) into N*K*2 bytes of fp16
 * 16 KB tiles of 128 rows x 64 columns, tile (n/128, k/64) at byte
 * ((n/128)*(K/64) + k/64)*16384, each stored as the 128-byte-swizzled K-major image the
 * tensor cores read from shared memory (bf16 values are exact in fp16 down to 2^-14 in
 * magnitude; smaller ones keep 2^-24 absolute precision). pic_model_create does this for
 * every bf16 projection matrix (one library-owned copy) so each weight tile streams from
 * HBM as one sequential bulk copy and the activations can be fp16. */
pic_status pic_op_pack_weight(const void* W, void* out, int32_t N, int32_t K, pic_stream_t stream);
/* Y[T][N] (fp32, overwritten) = X[T][K] . W^T with W in the pic_op_pack_weight layout and
 * X fp16, on the tcgen05 kernel. */
pic_status pic_op_gemm_packed(const void* W_packed, const void* X, float* Y, int32_t N, int32_t K, int32_t T,
                              pic_stream_t stream);

/* Sparse-query paged attention with fused RoPE for ONE sequence of pages:
 * out[t][h] = softmax_u( RoPE(q[t][h], q_pos[t]) . RoPE(K[u][g], pos(u)) / sqrt(D) ) V[u][g]
 * over every key u of the listed pages with pos(u) <= q_pos[t], g = h / (H/G).
 * dtype: type of the K/V pools. q: fp32 [T][H][D] (pre-RoPE); out: [T][H][D] fp16 when
 * dtype is PIC_BF16 (the operand type of the projection that follows), fp32 when PIC_F32.
 * q_pos: HOST [T] (ascending); pages: HOST arrays of n_pages (block, position of row 0,
 * valid rows); k_layer/v_layer: one layer of the pools ([pool_blocks][G][16][D]); every
 * page block must be < pool_blocks. rope_cs: device float2 [rope_positions][D/2] (cos,
 * sin), e.g. from pic_op_rope_table; every position must be < rope_positions, and
 * rope_positions >= 16. Scratch as reported by pic_op_attention_scratch_bytes (the work
 * list, split partials, and for the tensor-core path -- bf16, head_dim 128, 4 query heads
 * per KV head -- q and every page's K rotated to fp16). Rows beyond a page's length are
 * never read. */
size_t pic_op_attention_scratch_bytes(int32_t T, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                      int32_t n_pages);
pic_status pic_op_attention(int32_t dtype, int32_t T, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                            const void* q, const int32_t* q_pos_host, const void* k_layer, const void* v_layer,
                            const int32_t* page_block_host, const int32_t* page_pos_host,
                            const int32_t* page_len_host, int32_t n_pages, int32_t pool_blocks,
                            const void* rope_cs, int32_t rope_positions, void* out, void* scratch,
                            size_t scratch_bytes, pic_stream_t stream);

/* Allocation-free twin of pic_op_attention. The pages have no counterpart for this
 * call: it exists for callers that cannot allocate device memory (code running inside
 * a memory pool it does not own, plug-ins of hosts that forbid cudaMalloc after
 * start-up, paths that must not synchronize the device). Arguments and results are
 * those of pic_op_attention without the scratch buffer: the call uses a fixed 16 MiB
 * area inside the library (pic_op_attention_noalloc_max_scratch() bytes), held by every
 * GPU that loads the library until the process exits. It calls no cudaMalloc/cudaFree.
 *  - A shape whose exact work list, partial results and (tensor-core path) rotated q
 *    and K exceed the area is rejected with PIC_ERR_CAPACITY before any GPU work.
 *  - The first call on a device looks up the area's device address (with that device
 *    current). That look-up is guarded by a lock, so first calls from several host
 *    threads are safe.
 *  - Every call reuses the same area and leaves its contents behind; nothing in it has
 *    to start at zero (each word read is written earlier in the same call). Calls that
 *    overlap on the GPU (different streams, or different host threads) race on it:
 *    order them, e.g. by issuing them on one stream. */
size_t pic_op_attention_noalloc_max_scratch(void);
pic_status pic_op_attention_noalloc(int32_t dtype, int32_t T, int32_t n_heads, int32_t n_kv_heads,
                                    int32_t head_dim, const void* q, const int32_t* q_pos_host,
                                    const void* k_layer, const void* v_layer, const int32_t* page_block_host,
                                    const int32_t* page_pos_host, const int32_t* page_len_host, int32_t n_pages,
                                    int32_t pool_blocks, const void* rope_cs, int32_t rope_positions, void* out,
                                    pic_stream_t stream);

/* Host only (no GPU work, no device needed): the attention work plan the library launches
 * for a batch of sequences, e.g. the requests of a link or a decode step, each with its
 * selected rows and its pages. Rows are grouped in blocks of up to 64 (tensor-core shape:
 * bf16, head_dim 128, 4 query heads per KV head), 32 (mma.sync shapes with up to 4 query
 * heads per KV head) or 16 consecutive rows of one sequence; a block reads its sequence's
 * pages up to the page holding its last row's position, split into runs ("parts") whose
 * partial results are merged per (block, KV head).
 * seq_rows, seq_pages: [n_seqs + 1] non-decreasing offsets into row_pos [seq_rows[n_seqs]]
 * and page_pos [seq_pages[n_seqs]] (positions ascending within each sequence); num_sms >= 1.
 * Outputs (host): items [max_items][7] = (row0, nrows, kv_head, page0, page1, part,
 * page_mid), part -1 when the block's pages are not split, page_mid the end of the pages of
 * [page0, page1) that the item's first 32 rows can see (page1 for items of <= 32 rows), in
 * the order the kernels take them (the persistent
 * kernel's CTA c of n = min(items, num_sms) takes items c, c + n, ...); combines
 * [max_combines][5] = (row0, nrows, kv_head, part0, nparts); counts [3] = (items, combines,
 * parts). PIC_ERR_CAPACITY when an output array is too small (counts are still set);
 * PIC_ERR_INVALID_ARG for inconsistent offsets or unordered positions. */
pic_status pic_op_attention_plan(int32_t dtype, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                 int32_t n_seqs, const int32_t* seq_rows, const int32_t* seq_pages,
                                 const int32_t* row_pos, const int32_t* page_pos, int32_t num_sms, int32_t* items,
                                 int32_t max_items, int32_t* combines, int32_t max_combines, int32_t* counts);

/* Fills a device float2 table [n_pos][head_dim/2] with (cos, sin)(p * base^(-2i/D)),
 * angles formed in fp64 on the host. */
pic_status pic_op_rope_table(int32_t n_pos, int32_t head_dim, double base, void* out, pic_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PIC_H_ */
