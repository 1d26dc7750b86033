"""Python binding over the C ABI. PyTorch supplies device memory and streams; every
step of compile and link runs in the library's CUDA kernels. This module only
marshals arguments (pointers, sizes, host arrays) and keeps borrowed tensors alive.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import _lib as L

BLOCK = 16


def _stream(stream: Optional[torch.cuda.Stream]) -> C.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(L.PI32)


def _dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return L.PIC_F32
    if dtype == torch.bfloat16:
        return L.PIC_BF16
    raise ValueError(f"unsupported dtype {dtype}")


class PicModel:
    """Model weights (device, borrowed by the library) and their C handle.

    `cfg` is any object with n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim,
    vocab, rope_base, rms_eps and dtype ('f32'/'bf16'). `weights` maps the names
    'embed', 'lm_head', 'final_norm', 'layers.{l}.{attn_norm,wq,wk,wv,wo,mlp_norm,w_gate,w_up,w_down}'
    to tensors in nn.Linear layout. The fused Q|K|V and gate|up matrices the library
    reads are laid out here once (a copy on the device).
    """

    def __init__(self, cfg, weights: Dict[str, torch.Tensor], device: str = "cuda"):
        self.lib = L.load()
        self.cfg = cfg
        self.dtype = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
        dev = torch.device(device)
        cast = lambda t: t.to(device=dev, dtype=self.dtype).contiguous()
        self.t: Dict[str, torch.Tensor] = {
            "embed": cast(weights["embed"]), "lm_head": cast(weights["lm_head"]),
            "final_norm": weights["final_norm"].to(device=dev, dtype=torch.float32).contiguous()}
        for l in range(cfg.n_layers):
            p = f"layers.{l}."
            self.t[p + "attn_norm"] = weights[p + "attn_norm"].to(device=dev, dtype=torch.float32).contiguous()
            self.t[p + "mlp_norm"] = weights[p + "mlp_norm"].to(device=dev, dtype=torch.float32).contiguous()
            self.t[p + "w_qkv"] = torch.cat([cast(weights[p + n]) for n in ("wq", "wk", "wv")], 0).contiguous()
            self.t[p + "wo"] = cast(weights[p + "wo"])
            self.t[p + "w_gate_up"] = torch.cat([cast(weights[p + "w_gate"]), cast(weights[p + "w_up"])], 0).contiguous()
            self.t[p + "w_down"] = cast(weights[p + "w_down"])
        self._build()

    def _build(self):
        cfg = self.cfg
        c = L.ModelConfig(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                          cfg.vocab, float(cfg.rope_base), float(cfg.rms_eps), _dtype_code(self.dtype), BLOCK)
        nl = cfg.n_layers
        arr = lambda key: (C.c_void_p * nl)(*[self.t[f"layers.{l}.{key}"].data_ptr() for l in range(nl)])
        self._arrays = {k: arr(k) for k in ("attn_norm", "mlp_norm", "w_qkv", "wo", "w_gate_up", "w_down")}
        cast = lambda a: C.cast(a, C.POINTER(C.c_void_p))
        w = L.Weights(self.t["embed"].data_ptr(), self.t["lm_head"].data_ptr(), self.t["final_norm"].data_ptr(),
                      cast(self._arrays["attn_norm"]), cast(self._arrays["mlp_norm"]), cast(self._arrays["w_qkv"]),
                      cast(self._arrays["wo"]), cast(self._arrays["w_gate_up"]), cast(self._arrays["w_down"]))
        h = C.c_void_p()
        L.check(self.lib.pic_model_create(C.byref(c), C.byref(w), C.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.pic_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LinkResult:
    def __init__(self, hidden, logits, requests):
        self.hidden = hidden          # [sum Lq, d] fp32 (device)
        self.logits = logits          # [n_reqs or sum Lq, vocab] fp32 (device)
        self.requests = requests      # request handles


class DecodeResult:
    def __init__(self, hidden, logits, positions, slots):
        self.hidden = hidden          # [n, d] fp32 (device)
        self.logits = logits          # [n, vocab] fp32 (device)
        self.positions = positions    # int32 [n]: absolute position of each new token
        self.slots = slots            # int32 [n]: block_id * 16 + row of each new token


class PicStore:
    """Paged chunk-KV store: caller-owned pools (torch) + library-owned workspace."""

    def __init__(self, model: PicModel, num_blocks: int, max_rows: int, max_requests: int, max_positions: int,
                 max_logit_rows: int = 64, device: str = "cuda"):
        self.lib = model.lib
        self.model = model
        cfg = model.cfg
        self.num_blocks = num_blocks
        shape = (cfg.n_layers, num_blocks + 1, cfg.n_kv_heads, BLOCK, cfg.head_dim)
        self.k_pool = torch.zeros(shape, dtype=model.dtype, device=device)
        self.v_pool = torch.zeros(shape, dtype=model.dtype, device=device)
        sc = L.StoreConfig(num_blocks, max_rows, max_requests, max_positions, max_logit_rows)
        h = C.c_void_p()
        L.check(self.lib.pic_store_create(model.handle, C.byref(sc), self.k_pool.data_ptr(), self.v_pool.data_ptr(),
                                          C.byref(h)))
        self.handle = h
        self.max_logit_rows = max_logit_rows
        self._chunk_len = {}   # chunk handle -> tokens (sizes the optional scores output)

    # -- compile / import
    def compile(self, chunks: Sequence[np.ndarray], n_dummy: int = 0, stream=None) -> List[int]:
        toks = [_i32(c) for c in chunks]
        ptrs = (L.PI32 * len(toks))(*[_ptr_i32(t) for t in toks])
        lens = _i32([len(t) for t in toks])
        out = np.zeros(len(toks), dtype=np.int32)
        L.check(self.lib.pic_compile(self.handle, ptrs, _ptr_i32(lens), len(toks), n_dummy, _stream(stream),
                                     _ptr_i32(out)))
        self._chunk_len.update(zip(out.tolist(), (len(t) for t in toks)))
        return out.tolist()

    def import_chunk(self, tokens: np.ndarray, k: torch.Tensor, v: torch.Tensor, stream=None) -> int:
        """k, v: device [n_layers, n, G, D] pre-RoPE KV in the model dtype."""
        t = _i32(tokens)
        k = k.contiguous()
        v = v.contiguous()
        out = np.zeros(1, dtype=np.int32)
        L.check(self.lib.pic_chunk_import(self.handle, _ptr_i32(t), len(t), k.data_ptr(), v.data_ptr(),
                                          _stream(stream), _ptr_i32(out)))
        self._chunk_len[int(out[0])] = len(t)
        return int(out[0])

    # -- link
    def _link_args(self, requests, all_logits, hidden_out, logits_out):
        cfg = self.model.cfg
        keep = []
        reqs = (L.LinkRequest * len(requests))()
        n_q = 0
        for i, (cids, q) in enumerate(requests):
            ca, qa = _i32(cids), _i32(q)
            keep += [ca, qa]
            reqs[i] = L.LinkRequest(_ptr_i32(ca), len(ca), _ptr_i32(qa), len(qa))
            n_q += len(qa)
        n_lg = n_q if all_logits else len(requests)
        dev = self.k_pool.device
        if hidden_out is None:
            hidden_out = torch.empty((n_q, cfg.d_model), dtype=torch.float32, device=dev)
        if logits_out is None:
            logits_out = torch.empty((n_lg, cfg.vocab), dtype=torch.float32, device=dev)
        assert hidden_out.shape == (n_q, cfg.d_model) and hidden_out.dtype == torch.float32
        assert logits_out.shape == (n_lg, cfg.vocab) and logits_out.dtype == torch.float32
        return reqs, keep, hidden_out, logits_out

    def link(self, requests: Sequence[Tuple[Sequence[int], np.ndarray]], k: int, all_logits: bool = False,
             stream=None, hidden_out: Optional[torch.Tensor] = None,
             logits_out: Optional[torch.Tensor] = None) -> LinkResult:
        """pic_link (LegoLink-k): the first k tokens of every chunk and the query recomputed."""
        reqs, keep, hidden_out, logits_out = self._link_args(requests, all_logits, hidden_out, logits_out)
        out = np.zeros(len(requests), dtype=np.int32)
        L.check(self.lib.pic_link(self.handle, reqs, len(requests), k, int(all_logits), hidden_out.data_ptr(),
                                  logits_out.data_ptr(), _stream(stream), _ptr_i32(out)))
        return LinkResult(hidden_out, logits_out, out.tolist())

    def link_dynamic(self, requests: Sequence[Tuple[Sequence[int], np.ndarray]], r_percent: int,
                     all_logits: bool = False, stream=None, hidden_out: Optional[torch.Tensor] = None,
                     logits_out: Optional[torch.Tensor] = None, scores_out: Optional[torch.Tensor] = None
                     ) -> LinkResult:
        """pic_link_dynamic (CacheBlend-r): the r % prompt tokens the query attends to most at
        layer 0, and the query, recomputed. scores_out: optional device fp32 [sum of prompt
        lengths] receiving the token scores."""
        reqs, keep, hidden_out, logits_out = self._link_args(requests, all_logits, hidden_out, logits_out)
        if scores_out is not None:
            n_tok = sum(self._chunk_len[c] for cids, _ in requests for c in cids)
            assert scores_out.shape == (n_tok,) and scores_out.dtype == torch.float32 and scores_out.is_cuda
        out = np.zeros(len(requests), dtype=np.int32)
        L.check(self.lib.pic_link_dynamic(self.handle, reqs, len(requests), int(r_percent), int(all_logits),
                                          hidden_out.data_ptr(), logits_out.data_ptr(),
                                          scores_out.data_ptr() if scores_out is not None else None,
                                          _stream(stream), _ptr_i32(out)))
        return LinkResult(hidden_out, logits_out, out.tolist())

    def compile_cached(self, chunks: Sequence[np.ndarray], n_dummy: int = 0, stream=None):
        """pic_compile_cached: (chunk handles, hit flags) -- a chunk whose content an earlier
        compile_cached already made resident is reused instead of compiled."""
        toks = [_i32(c) for c in chunks]
        ptrs = (L.PI32 * len(toks))(*[_ptr_i32(t) for t in toks])
        lens = _i32([len(t) for t in toks])
        out = np.zeros(len(toks), dtype=np.int32)
        hits = np.zeros(len(toks), dtype=np.int32)
        L.check(self.lib.pic_compile_cached(self.handle, ptrs, _ptr_i32(lens), len(toks), n_dummy, _stream(stream),
                                            _ptr_i32(out), _ptr_i32(hits)))
        self._chunk_len.update(zip(out.tolist(), (len(t) for t in toks)))
        return out.tolist(), hits.astype(bool).tolist()

    def cache_stats(self) -> Dict[str, int]:
        st = L.CacheStats()
        L.check(self.lib.pic_store_get_cache_stats(self.handle, C.byref(st)))
        return {name: int(getattr(st, name)) for name, _ in L.CacheStats._fields_}

    def evict(self, max_chunks: int = -1) -> int:
        """Evicts up to max_chunks (all when < 0) unreferenced cached chunks; returns how many."""
        n = C.c_int32()
        L.check(self.lib.pic_store_evict(self.handle, max_chunks, C.byref(n)))
        return n.value

    def decode(self, requests: Sequence[int], tokens: Sequence[int], stream=None,
               hidden_out: Optional[torch.Tensor] = None,
               logits_out: Optional[torch.Tensor] = None) -> DecodeResult:
        """One generated token per linked request (pic_decode): hidden [n, d_model] and logits
        [n, vocab] of the new rows, with their positions and slots."""
        cfg = self.model.cfg
        ra, ta = _i32(requests), _i32(tokens)
        n = len(ra)
        assert len(ta) == n
        dev = self.k_pool.device
        if hidden_out is None:
            hidden_out = torch.empty((n, cfg.d_model), dtype=torch.float32, device=dev)
        if logits_out is None:
            logits_out = torch.empty((n, cfg.vocab), dtype=torch.float32, device=dev)
        assert hidden_out.shape == (n, cfg.d_model) and hidden_out.dtype == torch.float32
        assert logits_out.shape == (n, cfg.vocab) and logits_out.dtype == torch.float32
        positions, slots = np.zeros(n, dtype=np.int32), np.zeros(n, dtype=np.int32)
        L.check(self.lib.pic_decode(self.handle, _ptr_i32(ra), _ptr_i32(ta), n, hidden_out.data_ptr(),
                                    logits_out.data_ptr(), _stream(stream), _ptr_i32(positions), _ptr_i32(slots)))
        return DecodeResult(hidden_out, logits_out, positions, slots)

    # -- metadata / lifetime
    def request_info(self, r: int) -> Dict[str, np.ndarray]:
        info = L.RequestInfo()
        L.check(self.lib.pic_request_get_info(self.handle, r, C.byref(info)))
        arr = lambda p, n: np.ctypeslib.as_array(p, shape=(n,)).copy() if n else np.zeros(0, dtype=np.int32)
        return {"selected": arr(info.selected, info.n_selected), "slots": arr(info.slots, info.n_selected),
                "page_table": arr(info.page_table, info.n_pages), "page_pos": arr(info.page_pos, info.n_pages),
                "page_len": arr(info.page_len, info.n_pages),
                "private_blocks": arr(info.private_blocks, info.n_private)}

    def chunk_blocks(self, c: int) -> np.ndarray:
        n = C.c_int32()
        p = L.PI32()
        L.check(self.lib.pic_chunk_get_blocks(self.handle, c, C.byref(n), C.byref(p)))
        return np.ctypeslib.as_array(p, shape=(n.value,)).copy() if n.value else np.zeros(0, dtype=np.int32)

    def release_chunk(self, c: int):
        L.check(self.lib.pic_release_chunk(self.handle, c))

    def release_request(self, r: int):
        L.check(self.lib.pic_release_request(self.handle, r))

    def free_blocks(self) -> int:
        return int(self.lib.pic_store_free_blocks(self.handle))

    def profile_begin(self):
        L.check(self.lib.pic_profile_begin(self.handle))

    def profile_end(self) -> Dict[str, Dict[str, float]]:
        """Per kernel class: launches, summed event ms, algorithmic bytes and FLOPs."""
        p = L.Profile()
        L.check(self.lib.pic_profile_end(self.handle, C.byref(p)))
        names = ["gemm", "attention", "rowwise", "copy", "gemm_gate_up", "select"]
        out = {n: {"launches": int(p.launches[i]), "ms": p.ms[i], "bytes": p.bytes[i], "flops": p.flops[i]}
               for i, n in enumerate(names)}
        out["total_launches"] = int(p.total_launches)
        return out

    def launch_count(self) -> int:
        return int(self.lib.pic_store_launch_count(self.handle))

    def sync(self, stream=None):
        L.check(self.lib.pic_sync(self.handle, _stream(stream)))

    def kv_rows(self, layer: int, slots: np.ndarray) -> Tuple[torch.Tensor, torch.Tensor]:
        """K and V rows [n, G, D] stored at the given slots of one layer (a device gather)."""
        s = torch.as_tensor(_i32(slots), device=self.k_pool.device, dtype=torch.long)
        kp, vp = self.k_pool[layer], self.v_pool[layer]
        return kp[s // BLOCK, :, s % BLOCK, :], vp[s // BLOCK, :, s % BLOCK, :]

    def close(self):
        if getattr(self, "handle", None):
            self.lib.pic_store_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------------------------------- kernel-level calls

def gemm(W: torch.Tensor, X: torch.Tensor, stream=None) -> torch.Tensor:
    """Y[T][N] = X[T][K] @ W[N][K]^T through pic_op_gemm (fp32 result)."""
    lib = L.load()
    N, K = W.shape
    T = X.shape[0]
    assert X.shape[1] == K and W.dtype == X.dtype and W.is_contiguous() and X.is_contiguous()
    dt = _dtype_code(W.dtype)
    Y = torch.empty((T, N), dtype=torch.float32, device=W.device)
    L.check(lib.pic_op_gemm(dt, W.data_ptr(), X.data_ptr(), Y.data_ptr(), N, K, T, _stream(stream)))
    return Y


def pack_weight(W: torch.Tensor, stream=None) -> torch.Tensor:
    """bf16 [N][K] -> the fp16 tensor-core tile layout (pic_op_pack_weight), as a flat tensor."""
    lib = L.load()
    N, K = W.shape
    out = torch.empty(N * K, dtype=torch.float16, device=W.device)
    L.check(lib.pic_op_pack_weight(W.contiguous().data_ptr(), out.data_ptr(), N, K, _stream(stream)))
    return out


def gemm_packed(Wp: torch.Tensor, N: int, K: int, X: torch.Tensor, stream=None) -> torch.Tensor:
    """Y[T][N] = X @ W^T with W in the pic_op_pack_weight layout (fp16 tiles) and X fp16."""
    lib = L.load()
    T = X.shape[0]
    assert X.dtype == torch.float16
    Y = torch.empty((T, N), dtype=torch.float32, device=X.device)
    L.check(lib.pic_op_gemm_packed(Wp.data_ptr(), X.contiguous().data_ptr(), Y.data_ptr(), N, K, T, _stream(stream)))
    return Y


def rope_table(n_pos: int, head_dim: int, base: float, device="cuda") -> torch.Tensor:
    lib = L.load()
    out = torch.empty((n_pos, head_dim // 2, 2), dtype=torch.float32, device=device)
    L.check(lib.pic_op_rope_table(n_pos, head_dim, float(base), out.data_ptr(), _stream(None)))
    return out


def attention(q: torch.Tensor, q_pos: np.ndarray, k_layer: torch.Tensor, v_layer: torch.Tensor,
              pages: Tuple[np.ndarray, np.ndarray, np.ndarray], rope: torch.Tensor, n_kv_heads: int,
              stream=None) -> torch.Tensor:
    """Paged attention of one sequence through pic_op_attention.

    q: fp32 [T, H, D] (pre-RoPE); k_layer/v_layer: one layer of the pools. Returns fp16
    [T, H, D] for bf16 pools, fp32 for fp32 pools.
    """
    lib = L.load()
    T, H, D = q.shape
    assert q.dtype == torch.float32
    blk, ppos, plen = (_i32(a) for a in pages)
    qp = _i32(q_pos)
    out = torch.empty(q.shape, dtype=torch.float16 if k_layer.dtype == torch.bfloat16 else torch.float32,
                      device=q.device)
    nb = lib.pic_op_attention_scratch_bytes(T, H, n_kv_heads, D, len(blk))
    scratch = torch.empty(max(nb, 1), dtype=torch.uint8, device=q.device)
    L.check(lib.pic_op_attention(_dtype_code(k_layer.dtype), T, H, n_kv_heads, D, q.contiguous().data_ptr(),
                                 _ptr_i32(qp), k_layer.data_ptr(), v_layer.data_ptr(), _ptr_i32(blk), _ptr_i32(ppos),
                                 _ptr_i32(plen), len(blk), k_layer.shape[0], rope.data_ptr(), rope.shape[0],
                                 out.data_ptr(), scratch.data_ptr(), nb, _stream(stream)))
    return out


def attention_plan(dtype: torch.dtype, n_heads: int, n_kv_heads: int, head_dim: int,
                   seqs: Sequence[Tuple[Sequence[int], Sequence[int]]], num_sms: int):
    """The attention work plan the library launches (pic_op_attention_plan; host only).

    seqs: per sequence (row positions, page start positions), both ascending. Returns
    (items int32 [n, 7] = row0, nrows, kv_head, page0, page1, part, page_mid; combines int32 [m, 5] =
    row0, nrows, kv_head, part0, nparts; number of parts), rows and pages indexed over the
    concatenation of the sequences.
    """
    lib = L.load()
    rows = [_i32(r) for r, _ in seqs]
    pages = [_i32(p) for _, p in seqs]
    seq_rows = _i32(np.concatenate([[0], np.cumsum([len(r) for r in rows])]))
    seq_pages = _i32(np.concatenate([[0], np.cumsum([len(p) for p in pages])]))
    rp = _i32(np.concatenate(rows)) if rows else _i32([])
    pp = _i32(np.concatenate(pages)) if pages else _i32([])
    counts = np.zeros(3, dtype=np.int32)
    cap_i, cap_c = 1024, 256
    while True:
        items = np.zeros((cap_i, 7), dtype=np.int32)
        combs = np.zeros((cap_c, 5), dtype=np.int32)
        st = lib.pic_op_attention_plan(_dtype_code(dtype), n_heads, n_kv_heads, head_dim, len(seqs), _ptr_i32(seq_rows),
                                       _ptr_i32(seq_pages), _ptr_i32(rp), _ptr_i32(pp), num_sms, _ptr_i32(items),
                                       cap_i, _ptr_i32(combs), cap_c, _ptr_i32(counts))
        if st == L.PIC_ERR_CAPACITY and (counts[0] > cap_i or counts[1] > cap_c):
            cap_i, cap_c = max(cap_i, int(counts[0])), max(cap_c, int(counts[1]))
            continue
        L.check(st)
        return items[:counts[0]].copy(), combs[:counts[1]].copy(), int(counts[2])
