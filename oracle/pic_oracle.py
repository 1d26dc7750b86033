"""fp64 CPU oracle for position-independent context caching (compile / LegoLink link).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's CPU
baseline may import this module. The product path (the CUDA library and its Python
binding) never calls it, and it never calls the product: the two share no code.

Sources (cited by page title and section):
  [EPIC-sum]  "EPIC: Efficient Position-Independent Caching for Serving Large
              Language Models", AI summary page on atlas.scime.ai: summary line,
              Approach, Measured effects table, Surprising findings.
  [EPIC-abs]  the same paper's English abstract (shd-paper.top entry for 2410.15332v3).
  [MEPIC]     "MEPIC: Memory Efficient Position Independent Caching for LLM Serving",
              abstract (searcharxiv.org/abs/2512.16822).

What the pages fix:
  * PIC is split into a compile step and a link step [EPIC-sum, summary line].
  * compile: each immutable chunk is prefilled on its own with position ids starting
    at zero [EPIC-sum, Approach].
  * link (LegoLink-k): recompute only the first k tokens of every chunk (static
    selection) so they stop acting as attention sinks; cost grows with the number of
    chunks [EPIC-sum, Approach; EPIC-abs].
  * LegoLink-0: prepend four dummy tokens at compile, discard their KV, recompute
    nothing at link [EPIC-sum, Measured effects table and Surprising findings].
  * paged storage: chunk KV starts on a page boundary, only the first block of a chunk
    is request specific, K is stored without positional encoding and RoPE is applied
    inside attention [MEPIC].

What the pages leave open and this oracle reads plainly (each reading is one line):
  * model: Llama-style pre-norm decoder; RMSNorm (eps from the spec, gains given),
    no biases, rotate-half RoPE with theta_i = base^(-2i/D), GQA with contiguous head
    groups, SwiGLU MLP, final RMSNorm, untied LM head.
  * positions after linking are contiguous: chunk i occupies o_i..o_i+L_i-1 and the
    query follows the last chunk; a row attends to every row with position <= its own.
  * k_i = min(k, L_i); chunk 1 is recomputed too.
  * LegoLink-0 dummies are token id 0 at positions 0..3; the chunk sits at 4..L+3
    during compile and at o_i.. after linking (K is stored pre-RoPE).
  * block ids: lowest free id first; compile takes ceil(L/16) ids; link takes, per
    request in order and per chunk in order, ceil(k_i/16) private ids, then
    ceil(Lq/16) query ids; allocation is all-or-nothing.
  * a private block is a copy of the chunk's shared block with its first k_i rows
    replaced by the recomputed rows.
  * outputs: final-normed hidden states of all query rows, logits of the last query
    row of each request (or of all query rows).
  * decode after link: one new token per request at the next position, run through
    every layer while attending to the request's whole linked KV (compiled rows, the
    recomputed rows that replaced them, the query rows and earlier decoded rows) and
    to itself; its pre-RoPE K/V go into the request's last page, or into a new block
    (lowest free id) when that page is full.

Everything is numpy float64. Weights and stored KV arrive as bf16/fp32 values and are
upcast exactly.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

BLOCK = 16


# --------------------------------------------------------------------------- model pieces

def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/D), i < D/2 (rotate-half pairing of dims i and i + D/2)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return base ** (-2.0 * i / head_dim)


def rope(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate x[n, heads, D] at integer positions pos[n]: pair (i, i+D/2) turns by pos*theta_i.

    RoPE is applied at attention time from each row's absolute position [MEPIC].
    """
    D = x.shape[-1]
    ang = np.outer(pos.astype(np.float64), rope_inv_freq(D, base))      # [n, D/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def causal_attention(q_rot: np.ndarray, k_rot: np.ndarray, v: np.ndarray,
                     q_pos: np.ndarray, k_pos: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(D), masked to k_pos <= q_pos) v, per head; GQA by contiguous groups.

    q_rot [n, H, D], k_rot/v [m, G, D] -> [n, H, D]. Q head h reads KV head h // (H/G).
    """
    n, H, D = q_rot.shape
    G = k_rot.shape[1]
    rep = H // G
    out = np.empty((n, H, D))
    allowed = k_pos[None, :] <= q_pos[:, None]                          # [n, m]
    scale = 1.0 / np.sqrt(D)
    for h in range(H):
        g = h // rep
        s = (q_rot[:, h, :] @ k_rot[:, g, :].T) * scale
        s = np.where(allowed, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out


def _f64(t) -> np.ndarray:
    """Exact upcast of a torch (bf16/fp32) or numpy array to float64."""
    if hasattr(t, "detach"):
        import torch
        return t.detach().to(torch.float64).cpu().numpy()
    return np.asarray(t, dtype=np.float64)


class OracleModel:
    """Weights upcast to fp64 one layer at a time (8B layers are ~1.75 GB in fp64)."""

    def __init__(self, spec, weights: Dict[str, object], cache_all: Optional[bool] = None):
        self.spec = spec
        self.w = weights
        self.cache_all = (spec.param_count() < 50_000_000) if cache_all is None else cache_all
        self._cache: Dict[int, Dict[str, np.ndarray]] = {}
        self.final_norm = _f64(weights["final_norm"])

    def layer(self, l: int) -> Dict[str, np.ndarray]:
        if l not in self._cache:
            if not self.cache_all:
                self._cache.clear()
            p = f"layers.{l}."
            self._cache[l] = {n: _f64(self.w[p + n]) for n in
                              ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")}
        return self._cache[l]

    def embed(self, tokens: np.ndarray) -> np.ndarray:
        import torch
        idx = torch.as_tensor(np.asarray(tokens, dtype=np.int64))
        return _f64(self.w["embed"][idx])

    def logits(self, x_normed: np.ndarray, block: int = 16384) -> np.ndarray:
        """x_normed [n, d] @ W_lm^T, W_lm upcast in vocabulary blocks."""
        W = self.w["lm_head"]
        V = W.shape[0]
        out = np.empty((x_normed.shape[0], V))
        for v0 in range(0, V, block):
            out[:, v0:v0 + block] = x_normed @ _f64(W[v0:v0 + block]).T
        return out


# --------------------------------------------------------------------------- sequence runner

@dataclasses.dataclass
class SeqJob:
    """One logical sequence: rows `sel` are (re)computed, all other rows reuse given KV.

    tokens:  int token ids of the whole sequence (positions 0..N-1, contiguous).
    sel:     ascending indices of the rows computed through every layer.
    base_kv: l -> (K, V) fp64 [N, G, D] pre-RoPE KV for the rows not in `sel`
             (rows in `sel` are ignored and replaced); None when every row is selected.
    Row r sits at position pos0 + r.
    """
    tokens: np.ndarray
    sel: np.ndarray
    base_kv: Optional[Callable[[int], Tuple[np.ndarray, np.ndarray]]] = None
    pos0: int = 0                  # position of row 0 (0 everywhere except the offset-invariance pin)


@dataclasses.dataclass
class SeqResult:
    hidden: np.ndarray                 # final-normed hidden of the selected rows [n_sel, d]
    k: List[np.ndarray]                # per layer recomputed pre-RoPE K of the selected rows [n_sel, G, D]
    v: List[np.ndarray]                # per layer recomputed V of the selected rows


def run_jobs(model: OracleModel, jobs: Sequence[SeqJob]) -> List[SeqResult]:
    """Layer-major forward of the selected rows of every job (weights upcast once per layer)."""
    sp = model.spec
    H, G, D = sp.n_heads, sp.n_kv_heads, sp.head_dim
    hs = [model.embed(np.asarray(j.tokens)[j.sel]) for j in jobs]
    ks: List[List[np.ndarray]] = [[] for _ in jobs]
    vs: List[List[np.ndarray]] = [[] for _ in jobs]
    for l in range(sp.n_layers):
        W = model.layer(l)
        for ji, job in enumerate(jobs):
            N = len(job.tokens)
            pos_all = np.arange(N) + job.pos0
            sel = np.asarray(job.sel)
            h = hs[ji]
            x = rms_norm(h, W["attn_norm"], sp.rms_eps)
            q = (x @ W["wq"].T).reshape(-1, H, D)
            k = (x @ W["wk"].T).reshape(-1, G, D)
            v = (x @ W["wv"].T).reshape(-1, G, D)
            ks[ji].append(k)
            vs[ji].append(v)
            if job.base_kv is None:
                assert len(sel) == N, "without reused KV every row must be selected"
                K_all, V_all = np.zeros((N, G, D)), np.zeros((N, G, D))
            else:
                K_all, V_all = (a.copy() for a in job.base_kv(l))
            K_all[sel] = k
            V_all[sel] = v
            qpos = sel + job.pos0
            att = causal_attention(rope(q, qpos, sp.rope_base), rope(K_all, pos_all, sp.rope_base),
                                   V_all, qpos, pos_all)
            h = h + att.reshape(len(sel), H * D) @ W["wo"].T
            x = rms_norm(h, W["mlp_norm"], sp.rms_eps)
            h = h + (silu(x @ W["w_gate"].T) * (x @ W["w_up"].T)) @ W["w_down"].T
            hs[ji] = h
    return [SeqResult(rms_norm(h, model.final_norm, sp.rms_eps), ks[i], vs[i]) for i, h in enumerate(hs)]


# --------------------------------------------------------------------------- reference steps

def full_prefill(model: OracleModel, tokens: np.ndarray) -> SeqResult:
    """Plain causal prefill of the whole sequence (the full-recompute baseline, FR)."""
    tokens = np.asarray(tokens)
    return run_jobs(model, [SeqJob(tokens, np.arange(len(tokens)))])[0]


def compile_chunks(model: OracleModel, chunks: Sequence[np.ndarray], n_dummy: int = 0,
                   dummy_token: int = 0) -> List[Tuple[List[np.ndarray], List[np.ndarray]]]:
    """Compile: prefill each chunk alone from position 0 and keep its pre-RoPE K and V.

    With n_dummy > 0 (LegoLink-0) the chunk is prefilled behind n_dummy dummy tokens and
    the dummy rows' KV is dropped. Returns per chunk (K per layer [L,G,D], V per layer).
    """
    jobs = []
    for c in chunks:
        seq = np.concatenate([np.full(n_dummy, dummy_token, dtype=np.int64), np.asarray(c, dtype=np.int64)])
        jobs.append(SeqJob(seq, np.arange(len(seq))))
    res = run_jobs(model, jobs)
    return [([k[n_dummy:] for k in r.k], [v[n_dummy:] for v in r.v]) for r in res]


# --------------------------------------------------------------------------- dynamic selection

def query_attention_scores(model: OracleModel, chunk_tokens: Sequence[np.ndarray], chunk_k0: Sequence[np.ndarray],
                           query: np.ndarray) -> np.ndarray:
    """Attention mass each prompt token receives from the query at layer 0 (dynamic selection).

    The pages compare LegoLink's static choice of chunk-initial tokens with CacheBlend's
    "dynamic attention-based selection" of the tokens to recompute (EPIC summary page:
    problem statement; Measured effects table, CacheBlend-r rows and the static-vs-dynamic
    row) without giving its formula. Reading: the prompt is linked with no recomputation
    (every chunk's compiled layer-0 K, rotated at its absolute position); the query rows'
    q and K are computed at layer 0; each query row and head attends causally over the
    prompt and the query; a prompt token's score is the sum of the softmax weights it gets
    over all query rows and heads. Returns scores [N] for the N prompt tokens.
    """
    sp = model.spec
    H, G, D = sp.n_heads, sp.n_kv_heads, sp.head_dim
    W = model.layer(0)
    q_tok = np.asarray(query)
    N = sum(len(t) for t in chunk_tokens)
    Lq = len(q_tok)
    x = rms_norm(model.embed(q_tok), W["attn_norm"], sp.rms_eps)
    q = (x @ W["wq"].T).reshape(Lq, H, D)
    kq = (x @ W["wk"].T).reshape(Lq, G, D)
    K = np.concatenate([_f64(k) for k in chunk_k0] + [kq])              # pre-RoPE, positions 0..N+Lq-1
    pos = np.arange(N + Lq)
    qpos = pos[N:]
    q_rot = rope(q, qpos, sp.rope_base)
    k_rot = rope(K, pos, sp.rope_base)
    allowed = pos[None, :] <= qpos[:, None]
    scores = np.zeros(N)
    rep = H // G
    for h in range(H):
        s = (q_rot[:, h, :] @ k_rot[:, h // rep, :].T) / np.sqrt(D)
        s = np.where(allowed, s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        scores += p[:, :N].sum(axis=0)
    return scores


def select_top(scores: np.ndarray, r_percent: int) -> np.ndarray:
    """The floor(r * N / 100) prompt positions with the largest scores (equal scores: the
    lower position first), in ascending position order (CacheBlend-r recomputes r % of the
    tokens: EPIC summary page, Measured effects table)."""
    N = len(scores)
    n = (int(r_percent) * N) // 100
    order = sorted(range(N), key=lambda u: (-scores[u], u))
    return np.asarray(sorted(order[:n]), dtype=np.int64)


# --------------------------------------------------------------------------- paged store

class OutOfBlocks(Exception):
    pass


@dataclasses.dataclass
class OracleChunk:
    tokens: np.ndarray
    blocks: List[int]
    k: List[np.ndarray]           # per layer pre-RoPE K [L, G, D] (fp64 or exact bf16 values)
    v: List[np.ndarray]
    refs: int = 1


@dataclasses.dataclass
class LinkMeta:
    """Integer metadata of one linked request (all int32, bit-exact contract)."""
    selected: np.ndarray          # absolute positions of recomputed rows, ascending
    slots: np.ndarray             # block_id * 16 + row for each selected row
    page_table: np.ndarray        # physical block ids in position order
    page_pos: np.ndarray          # absolute position of row 0 of each page
    page_len: np.ndarray          # valid rows in each page
    private_blocks: np.ndarray    # blocks this link allocated (chunk privates, then query)


@dataclasses.dataclass
class DecodeOut:
    """One decode step over a batch of linked requests."""
    positions: np.ndarray         # int32 [n]: absolute position of each new token
    slots: np.ndarray             # int32 [n]: block_id * 16 + row of each new token
    hidden: np.ndarray            # [n, d] final-normed hidden of the new rows
    logits: np.ndarray            # [n, vocab]
    k: List[List[np.ndarray]]     # per request, per layer pre-RoPE K of the new row [G, D]
    v: List[List[np.ndarray]]


@dataclasses.dataclass
class _LinkedKV:
    """What a decode step needs of a linked request: every token, and where each
    position's KV comes from (compiled chunk rows, overridden by the recomputed rows)."""
    chunk_ids: List[int]
    tokens: np.ndarray            # positions 0..N-1: chunks, query, decoded tokens
    selected: np.ndarray          # recomputed positions of the link
    k_sel: List[np.ndarray]       # per layer [n_sel, G, D]
    v_sel: List[np.ndarray]
    k_dec: List[List[np.ndarray]]  # per layer, the decoded rows' [G, D] in order
    v_dec: List[List[np.ndarray]]
    meta: LinkMeta                # page table of the request, grown by decode


@dataclasses.dataclass
class LinkOut:
    meta: List[LinkMeta]
    hidden: List[np.ndarray]      # per request final-normed hidden of the query rows [Lq, d]
    logits: List[np.ndarray]      # per request logits [1 or Lq, vocab]
    k: List[List[np.ndarray]]     # per request, per layer recomputed pre-RoPE K [n_sel, G, D]
    v: List[List[np.ndarray]]
    rids: List[int] = dataclasses.field(default_factory=list)   # request handles, for decode


class OracleStore:
    """The oracle's own block allocator, chunk table and link step."""

    def __init__(self, model: Optional[OracleModel], num_blocks: int):
        self.model = model
        self.num_blocks = num_blocks
        self.free = set(range(num_blocks))
        self.chunks: Dict[int, OracleChunk] = {}
        self.requests: Dict[int, Tuple[List[int], List[int]]] = {}
        self.linked: Dict[int, _LinkedKV] = {}
        self._next_chunk = 0
        self._next_req = 0

    # lowest-free-id allocator, all-or-nothing
    def _take(self, n: int) -> List[int]:
        if n > len(self.free):
            raise OutOfBlocks(f"need {n} blocks, {len(self.free)} free")
        ids = sorted(self.free)[:n]
        self.free.difference_update(ids)
        return ids

    def _add_chunk(self, tokens, k, v) -> int:
        blocks = self._take(-(-len(tokens) // BLOCK))
        cid = self._next_chunk
        self._next_chunk += 1
        self.chunks[cid] = OracleChunk(np.asarray(tokens, dtype=np.int64), blocks, k, v)
        return cid

    def compile(self, tokens: np.ndarray, n_dummy: int = 0) -> int:
        """Compile one chunk and store it in ceil(L/16) page-aligned blocks."""
        if -(-len(tokens) // BLOCK) > len(self.free):
            raise OutOfBlocks("compile")
        (k, v), = compile_chunks(self.model, [tokens], n_dummy)
        return self._add_chunk(tokens, k, v)

    def compile_many(self, chunks: Sequence[np.ndarray], n_dummy: int = 0) -> List[int]:
        need = sum(-(-len(c) // BLOCK) for c in chunks)
        if need > len(self.free):
            raise OutOfBlocks("compile")
        kv = compile_chunks(self.model, chunks, n_dummy)
        return [self._add_chunk(c, k, v) for c, (k, v) in zip(chunks, kv)]

    def import_chunk(self, tokens: np.ndarray, k_layers, v_layers) -> int:
        """Store externally produced chunk KV (per layer [L, G, D]) as if compiled.

        Values are kept as given (bf16/fp32 are exact in fp64) and upcast layer by layer
        when the link reads them.
        """
        return self._add_chunk(tokens, list(k_layers), list(v_layers))

    def release_chunk(self, cid: int) -> None:
        c = self.chunks[cid]
        c.refs -= 1
        if c.refs == 0:
            self.free.update(c.blocks)
            del self.chunks[cid]

    def release_request(self, rid: int) -> None:
        blocks, cids = self.requests.pop(rid)
        self.linked.pop(rid, None)
        self.free.update(blocks)
        for cid in cids:
            self.release_chunk(cid)

    # -- link metadata (steps a1-a3)
    def plan(self, requests: Sequence[Tuple[Sequence[int], int]], k: int) -> List[LinkMeta]:
        """Allocate private/query blocks and build page tables, selected rows and slots.

        requests: (chunk ids in prompt order, query length). Raises OutOfBlocks with no
        state change when the pool cannot hold every request's new blocks.
        """
        need = 0
        for cids, lq in requests:
            need += sum(-(-min(k, len(self.chunks[c].tokens)) // BLOCK) for c in cids) + (-(-lq // BLOCK))
        if need > len(self.free):
            raise OutOfBlocks("link")
        metas = []
        for cids, lq in requests:
            sel, slots, table, ppos, plen, priv = [], [], [], [], [], []
            off = 0
            for c in cids:
                ch = self.chunks[c]
                L = len(ch.tokens)
                ki = min(k, L)
                m = -(-ki // BLOCK)
                own = self._take(m)
                priv += own
                for j in range(-(-L // BLOCK)):
                    table.append(own[j] if j < m else ch.blocks[j])
                    ppos.append(off + BLOCK * j)
                    plen.append(min(BLOCK, L - BLOCK * j))
                for t in range(ki):
                    sel.append(off + t)
                    slots.append(own[t // BLOCK] * BLOCK + t % BLOCK)
                off += L
            qb = self._take(-(-lq // BLOCK))
            priv += qb
            for j in range(len(qb)):
                table.append(qb[j])
                ppos.append(off + BLOCK * j)
                plen.append(min(BLOCK, lq - BLOCK * j))
            for t in range(lq):
                sel.append(off + t)
                slots.append(qb[t // BLOCK] * BLOCK + t % BLOCK)
            i32 = lambda a: np.asarray(a, dtype=np.int32)
            metas.append(LinkMeta(i32(sel), i32(slots), i32(table), i32(ppos), i32(plen), i32(priv)))
        return metas

    def plan_selected(self, requests: Sequence[Tuple[Sequence[int], int, Sequence[Sequence[int]]]]) -> List[LinkMeta]:
        """Metadata of a link whose recomputed rows are given per chunk (dynamic selection).

        requests: (chunk ids, query length, per chunk the ascending token indices to
        recompute). Every block of a chunk that holds a recomputed token becomes the
        request's own copy (MEPIC abstract: only request-specific blocks are private); a
        request takes, per chunk in order, one new block per such chunk block in ascending
        order, then its query blocks; lowest free id first, all or nothing.
        """
        blocks_of = lambda sel: sorted({t // BLOCK for t in sel})
        need = 0
        for cids, lq, sels in requests:
            need += sum(len(blocks_of(sel)) for sel in sels) + (-(-lq // BLOCK))
        if need > len(self.free):
            raise OutOfBlocks("link")
        metas = []
        for cids, lq, sels in requests:
            sel, slots, table, ppos, plen, priv = [], [], [], [], [], []
            off = 0
            for c, cs in zip(cids, sels):
                ch = self.chunks[c]
                L = len(ch.tokens)
                mine = blocks_of(cs)
                own = dict(zip(mine, self._take(len(mine))))
                priv += [own[j] for j in mine]
                for j in range(-(-L // BLOCK)):
                    table.append(own.get(j, ch.blocks[j]))
                    ppos.append(off + BLOCK * j)
                    plen.append(min(BLOCK, L - BLOCK * j))
                for t in cs:
                    sel.append(off + t)
                    slots.append(own[t // BLOCK] * BLOCK + t % BLOCK)
                off += L
            qb = self._take(-(-lq // BLOCK))
            priv += qb
            for j in range(len(qb)):
                table.append(qb[j])
                ppos.append(off + BLOCK * j)
                plen.append(min(BLOCK, lq - BLOCK * j))
            for t in range(lq):
                sel.append(off + t)
                slots.append(qb[t // BLOCK] * BLOCK + t % BLOCK)
            i32 = lambda a: np.asarray(a, dtype=np.int32)
            metas.append(LinkMeta(i32(sel), i32(slots), i32(table), i32(ppos), i32(plen), i32(priv)))
        return metas

    def link_selected(self, requests: Sequence[Tuple[Sequence[int], np.ndarray, Sequence[Sequence[int]]]],
                      all_logits: bool = False) -> LinkOut:
        """Link with the recomputed rows given per chunk: the same steps as `link` (a4-a10)
        over those rows, metadata from `plan_selected`."""
        metas = self.plan_selected([(cids, len(q), sels) for cids, q, sels in requests])
        return self._run_link([(cids, q) for cids, q, _ in requests], metas, all_logits)

    def link_dynamic(self, requests: Sequence[Tuple[Sequence[int], np.ndarray]], r_percent: int,
                     all_logits: bool = False) -> Tuple[LinkOut, List[np.ndarray]]:
        """CacheBlend-r: per request, score the prompt tokens by the query's attention
        (`query_attention_scores`), recompute the top r % of them (`select_top`) and the
        query. Returns the link and each request's scores."""
        sels, scores = [], []
        for cids, q in requests:
            chs = [self.chunks[c] for c in cids]
            sc = query_attention_scores(self.model, [c.tokens for c in chs], [c.k[0] for c in chs], q)
            top = select_top(sc, r_percent)
            per, off = [], 0
            for c in chs:
                L = len(c.tokens)
                per.append([int(u - off) for u in top if off <= u < off + L])
                off += L
            sels.append(per)
            scores.append(sc)
        out = self.link_selected([(cids, q, sel) for (cids, q), sel in zip(requests, sels)], all_logits)
        return out, scores

    def link(self, requests: Sequence[Tuple[Sequence[int], np.ndarray]], k: int,
             all_logits: bool = False) -> LinkOut:
        """LegoLink-k over a batch of requests (steps a1-a10), returning outputs and metadata."""
        metas = self.plan([(cids, len(q)) for cids, q in requests], k)
        return self._run_link(requests, metas, all_logits)

    def _run_link(self, requests, metas: List[LinkMeta], all_logits: bool) -> LinkOut:
        """Steps a4-a10 of a link whose metadata (blocks taken, selected rows) is planned."""
        rids = []
        for (cids, _), meta in zip(requests, metas):
            rid = self._next_req
            self._next_req += 1
            for c in cids:
                self.chunks[c].refs += 1
            self.requests[rid] = (list(meta.private_blocks), list(cids))
            rids.append(rid)
        jobs = []
        for (cids, q), meta in zip(requests, metas):
            chs = [self.chunks[c] for c in cids]
            seq = np.concatenate([c.tokens for c in chs] + [np.asarray(q, dtype=np.int64)])
            lq = len(q)

            def base_kv(l, chs=chs, lq=lq):
                G, D = self.model.spec.n_kv_heads, self.model.spec.head_dim
                K = np.concatenate([_f64(c.k[l]) for c in chs] + [np.zeros((lq, G, D))])
                V = np.concatenate([_f64(c.v[l]) for c in chs] + [np.zeros((lq, G, D))])
                return K, V
            jobs.append(SeqJob(seq, meta.selected.astype(np.int64), base_kv))
        res = run_jobs(self.model, jobs)
        hidden, logits = [], []
        for (cids, q), r, job, meta, rid in zip(requests, res, jobs, metas, rids):
            hq = r.hidden[-len(q):]
            hidden.append(hq)
            logits.append(self.model.logits(hq if all_logits else hq[-1:]))
            nl = self.model.spec.n_layers
            own = LinkMeta(*(np.array(getattr(meta, f.name)) for f in dataclasses.fields(LinkMeta)))
            self.linked[rid] = _LinkedKV(list(cids), np.asarray(job.tokens), job.sel, r.k, r.v,
                                         [[] for _ in range(nl)], [[] for _ in range(nl)], own)
        return LinkOut(metas, hidden, logits, [r.k for r in res], [r.v for r in res], rids)

    def request_meta(self, rid: int) -> LinkMeta:
        """Current page table of a linked request (grows with every decoded token)."""
        return self.linked[rid].meta

    def _request_kv(self, rid: int, l: int) -> Tuple[np.ndarray, np.ndarray]:
        """Pre-RoPE K, V [N, G, D] of every position of a linked request at layer l: the
        compiled chunk rows, the link's recomputed rows in their place, then the query rows
        and the decoded rows."""
        st = self.linked[rid]
        G, D = self.model.spec.n_kv_heads, self.model.spec.head_dim
        N = len(st.tokens)
        K, V = np.zeros((N, G, D)), np.zeros((N, G, D))
        off = 0
        for c in st.chunk_ids:
            ch = self.chunks[c]
            L = len(ch.tokens)
            K[off:off + L] = _f64(ch.k[l])
            V[off:off + L] = _f64(ch.v[l])
            off += L
        K[st.selected] = st.k_sel[l]
        V[st.selected] = st.v_sel[l]
        n_dec = len(st.k_dec[l])
        if n_dec:
            K[N - n_dec:] = np.stack(st.k_dec[l])
            V[N - n_dec:] = np.stack(st.v_dec[l])
        return K, V

    def decode(self, rids: Sequence[int], tokens: Sequence[int]) -> DecodeOut:
        """One decode step: token tokens[i] is appended to linked request rids[i] at the
        position after its last one and run through every layer; it attends to all of the
        request's KV and to itself. A request whose last page is full first takes the
        lowest free block (all requests' blocks or none). Requests must be distinct."""
        rids = list(rids)
        if len(set(rids)) != len(rids) or len(tokens) != len(rids):
            raise ValueError("decode: one token per distinct request")
        need = sum(1 for rid in rids if self.linked[rid].meta.page_len[-1] == BLOCK)
        if need > len(self.free):
            raise OutOfBlocks("decode")
        positions, slots, jobs = [], [], []
        for rid, tok in zip(rids, tokens):
            st = self.linked[rid]
            m = st.meta
            pos = int(m.page_pos[-1]) + int(m.page_len[-1])
            if m.page_len[-1] == BLOCK:
                b, = self._take(1)
                self.requests[rid][0].append(b)
                m.page_table = np.append(m.page_table, np.int32(b))
                m.page_pos = np.append(m.page_pos, np.int32(pos))
                m.page_len = np.append(m.page_len, np.int32(1))
                m.private_blocks = np.append(m.private_blocks, np.int32(b))
            else:
                m.page_len[-1] += 1
            positions.append(pos)
            slots.append(int(m.page_table[-1]) * BLOCK + int(m.page_len[-1]) - 1)

            def base_kv(l, rid=rid):
                K, V = self._request_kv(rid, l)    # positions 0..pos-1; the new row is appended
                G, D = K.shape[1], K.shape[2]
                return np.concatenate([K, np.zeros((1, G, D))]), np.concatenate([V, np.zeros((1, G, D))])
            jobs.append(SeqJob(np.append(st.tokens, np.int64(tok)), np.array([pos]), base_kv))
        # every job reads its base KV before any new row is stored
        res = run_jobs(self.model, jobs)
        for rid, tok, r in zip(rids, tokens, res):
            st = self.linked[rid]
            st.tokens = np.append(st.tokens, np.int64(tok))
            for l in range(self.model.spec.n_layers):
                st.k_dec[l].append(r.k[l][0])
                st.v_dec[l].append(r.v[l][0])
        hidden = np.concatenate([r.hidden for r in res])
        i32 = lambda a: np.asarray(a, dtype=np.int32)
        return DecodeOut(i32(positions), i32(slots), hidden, self.model.logits(hidden),
                         [[k[0] for k in r.k] for r in res], [[v[0] for v in r.v] for r in res])
