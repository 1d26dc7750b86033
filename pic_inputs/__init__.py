"""Seeded synthetic inputs shared by the CUDA library's tests/bench and the CPU oracle.

This module only *draws* inputs: model shapes, random weights, token ids, request
mixes and stand-in compiled chunk KV. It holds none of the method's arithmetic
(no norm, projection, RoPE, attention or paging logic), so both sides can consume
the same values without sharing any computation.

Workload shapes follow the EPIC summary page (atlas.scime.ai, "EPIC: Efficient
Position-Independent Caching for Serving Large Language Models", Key results and
Measured effects table: 512-token chunks, k up to 32, LegoLink-0 with four dummy
tokens) and the MEPIC abstract (searcharxiv.org 2512.16822: 16-token pages, first
block request-specific). The model architecture is a Llama-style decoder because
the pages print none; the datasets the pages evaluate on (LongBench) are replaced
by uniform random token ids of the same chunk structure.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
import zlib
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

BLOCK_SIZE = 16          # tokens per KV page (MEPIC paged storage)
DUMMY_TOKEN = 0          # token id used for the LegoLink-0 dummy prefix
N_DUMMY_LEGOLINK0 = 4    # "prepend ... four dummy tokens" (EPIC summary, Measured effects table)

WEIGHT_SEED = 1234
TOKEN_SEED = 1
REQUEST_SEED = 2
KV_SEED = 3
QUERY_SEED = 4


@dataclasses.dataclass(frozen=True)
class ModelSpec:
    """Shape of a Llama-style pre-norm decoder (RMSNorm, RoPE, GQA, SwiGLU, untied head)."""
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_base: float
    rms_eps: float = 1e-5
    dtype: str = "f32"          # "f32" or "bf16": storage type of weights, KV and GEMM operands
    block_size: int = BLOCK_SIZE

    @property
    def qkv_dim(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_layers(self, n_layers: int) -> "ModelSpec":
        return dataclasses.replace(self, n_layers=n_layers, name=f"{self.name}-L{n_layers}")

    def param_count(self) -> int:
        d, f, v = self.d_model, self.ffn_dim, self.vocab
        per_layer = d * self.qkv_dim + self.n_heads * self.head_dim * d + 3 * d * f
        return self.n_layers * per_layer + 2 * v * d


# Tiny fp32 decoder: 2 layers, d 256, 4/4 heads, head_dim 64, ffn 512, vocab 1024, base 1e4.
TINY = ModelSpec("tiny-f32", 2, 256, 4, 4, 64, 512, 1024, 10000.0, 1e-5, "f32")
# Llama-3-8B shape, bf16, random init.
LLAMA3_8B = ModelSpec("llama3-8b-shape", 32, 4096, 32, 8, 128, 14336, 128256, 500000.0, 1e-5, "bf16")
# Very small GQA decoder used where brute-force loops must stay cheap (2 Q heads per KV head).
MICRO_GQA = ModelSpec("micro-gqa", 2, 64, 4, 2, 16, 96, 97, 10000.0, 1e-5, "f32")
# Small bf16 GQA decoder with head_dim 128 (exercises the bf16 kernels at small cost).
SMALL_BF16 = ModelSpec("small-bf16-gqa", 2, 512, 8, 2, 128, 1024, 2048, 500000.0, 1e-5, "bf16")


def _seed(*parts) -> int:
    """Stable 63-bit seed from a tuple of ints/strings (platform independent)."""
    words = []
    for p in parts:
        if isinstance(p, str):
            words.append(zlib.crc32(p.encode()))
        else:
            words.append(int(p) & 0xFFFFFFFF)
    ss = np.random.SeedSequence(words)
    return int(ss.generate_state(1, dtype=np.uint64)[0]) & ((1 << 63) - 1)


_POOL: Optional[_cf.ThreadPoolExecutor] = None


def _pool() -> _cf.ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = _cf.ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1)))
    return _POOL


_BLOCK = 1 << 23


def randn(shape: Sequence[int], seed: Tuple, std: float = 1.0,
          dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """N(0, std^2) draws, generated in independently seeded 8M-element blocks (threaded).

    The result depends only on (shape, seed, std, dtype), never on thread count.
    """
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=dtype)
    nblk = (n + _BLOCK - 1) // _BLOCK

    def fill(b):
        lo, hi = b * _BLOCK, min(n, (b + 1) * _BLOCK)
        g = torch.Generator().manual_seed(_seed(*seed, "blk", b))
        x = torch.randn(hi - lo, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[lo:hi] = x.to(dtype)

    if nblk <= 1:
        fill(0) if n else None
    else:
        list(_pool().map(fill, range(nblk)))
    return out.view(*shape)


# ----------------------------------------------------------------------------- weights

def layer_weight_names() -> List[str]:
    return ["attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"]


def weight_shape(spec: ModelSpec, name: str) -> Tuple[int, ...]:
    d, H, G, D, f = spec.d_model, spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.ffn_dim
    return {
        "embed": (spec.vocab, d), "lm_head": (spec.vocab, d), "final_norm": (d,),
        "attn_norm": (d,), "mlp_norm": (d,),
        "wq": (H * D, d), "wk": (G * D, d), "wv": (G * D, d), "wo": (d, H * D),
        "w_gate": (f, d), "w_up": (f, d), "w_down": (d, f),
    }[name]


def gen_weight(spec: ModelSpec, name: str, layer: int = -1, seed: int = WEIGHT_SEED,
               gains: str = "ones") -> torch.Tensor:
    """One weight tensor in nn.Linear layout ([out, in]).

    Matrices: N(0, 1/d_model) for every matrix (embedding and LM head included),
    stored in the spec's dtype. Norm gains: fp32, all ones ("ones") or 1 + 0.1*N(0,1)
    ("random", used by tests so that a dropped gain is visible).
    """
    shape = weight_shape(spec, name)
    if name.endswith("norm"):
        if gains == "ones":
            return torch.ones(shape, dtype=torch.float32)
        return 1.0 + randn(shape, (seed, spec.name, name, layer, "gain"), 0.1)
    std = 1.0 / float(np.sqrt(spec.d_model))
    return randn(shape, (seed, spec.name, name, layer), std, spec.torch_dtype)


def gen_weights(spec: ModelSpec, seed: int = WEIGHT_SEED, gains: str = "ones",
                layers: Optional[Sequence[int]] = None) -> Dict[str, torch.Tensor]:
    """All weights as a flat dict: 'embed', 'lm_head', 'final_norm', 'layers.{l}.{name}'."""
    w = {n: gen_weight(spec, n, -1, seed, gains) for n in ("embed", "lm_head", "final_norm")}
    for l in (range(spec.n_layers) if layers is None else layers):
        for n in layer_weight_names():
            w[f"layers.{l}.{n}"] = gen_weight(spec, n, l, seed, gains)
    return w


# ----------------------------------------------------------------------------- tokens / KV

def gen_tokens(n: int, vocab: int, *seed) -> np.ndarray:
    """Uniform token ids in [0, vocab) (stand-in for document text)."""
    rng = np.random.Generator(np.random.PCG64(_seed(*seed)))
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def gen_chunk_kv(spec: ModelSpec, n_tokens: int, chunk_seed: int, seed: int = KV_SEED):
    """Stand-in for a compiled chunk's KV: per layer pre-RoPE K and V [n_tokens, G, D] ~ N(0,1).

    The unit variance matches K/V = W x for an RMS-normalised x and W ~ N(0, 1/d).
    Returns (K, V) as tensors of shape [n_layers, n_tokens, G, D] in the spec's dtype.
    """
    shape = (spec.n_layers, n_tokens, spec.n_kv_heads, spec.head_dim)
    k = randn(shape, (seed, spec.name, "K", chunk_seed), 1.0, spec.torch_dtype)
    v = randn(shape, (seed, spec.name, "V", chunk_seed), 1.0, spec.torch_dtype)
    return k, v


def zipf_draws(n_draw: int, pool: int, s: float, *seed) -> List[int]:
    """n_draw distinct chunk ids from ranks 1..pool with P(r) ~ r^-s, then a random order.

    Rank r maps to chunk id r-1; duplicates are redrawn; the kept ids are permuted.
    """
    rng = np.random.Generator(np.random.PCG64(_seed(*seed)))
    p = np.arange(1, pool + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    picked: List[int] = []
    while len(picked) < n_draw:
        r = int(rng.choice(pool, p=p))
        if r not in picked:
            picked.append(r)
    perm = rng.permutation(n_draw)
    return [picked[i] for i in perm]


# ----------------------------------------------------------------------------- workloads

@dataclasses.dataclass
class Request:
    chunk_ids: List[int]           # indices into Workload.chunks, in prompt order
    query: np.ndarray              # int32 query-suffix tokens


@dataclasses.dataclass
class Workload:
    name: str
    spec: ModelSpec
    chunks: List[np.ndarray]       # int32 token arrays of the immutable chunks
    requests: List[Request]
    k: int                         # tokens recomputed at the start of every chunk
    n_dummy: int = 0               # dummy tokens prepended at compile (LegoLink-0 uses 4)

    @property
    def linked_tokens(self) -> int:
        return sum(sum(len(self.chunks[c]) for c in r.chunk_ids) + len(r.query) for r in self.requests)

    @property
    def selected_rows(self) -> int:
        return sum(sum(min(self.k, len(self.chunks[c])) for c in r.chunk_ids) + len(r.query)
                   for r in self.requests)


def make_workload(name: str, spec: ModelSpec, n_chunks: int, chunk_len, query_len: int, k: int,
                  n_requests: int = 1, pool: Optional[int] = None, per_request: Optional[int] = None,
                  zipf_s: float = 1.1, n_dummy: int = 0) -> Workload:
    """Chunks of uniform random tokens and requests over them.

    chunk_len may be an int or a list (ragged chunks). Without `pool`, each request
    links all n_chunks chunks in order. With `pool`, n_chunks = pool size and each
    request draws `per_request` chunks by Zipf(zipf_s) in a random order.
    """
    lens = [chunk_len] * n_chunks if isinstance(chunk_len, int) else list(chunk_len)
    chunks = [gen_tokens(L, spec.vocab, TOKEN_SEED, spec.name, "chunk", c) for c, L in enumerate(lens)]
    reqs = []
    for r in range(n_requests):
        if pool is None:
            ids = list(range(n_chunks))
        else:
            ids = zipf_draws(per_request, pool, zipf_s, REQUEST_SEED, spec.name, r)
        q = gen_tokens(query_len, spec.vocab, QUERY_SEED, spec.name, "query", r)
        reqs.append(Request(ids, q))
    return Workload(name, spec, chunks, reqs, k, n_dummy)


def config_workloads(spec_8b: ModelSpec = LLAMA3_8B) -> Dict[str, Workload]:
    """The evaluated workloads, keyed by shape: tiny (fp32, 4 x 64 + 16, k = 2), 8b_10x512 (10 x 512 +
    64 query, k = 16), 8b_98x512 (98 x 512 + 64, k = 16), 8b_32req (32 requests x 8 Zipf chunks of
    a 64-chunk pool + 32 query, k = 16) and the k sweep 8b_10x512_k{0,2,16,32,512} (k = 0 with
    the LegoLink-0 dummy prefix)."""
    w = {
        "tiny": make_workload("tiny: 4x64 + 16 query, k=2", TINY, 4, 64, 16, 2),
        "8b_10x512": make_workload("8B: 10x512 + 64 query, k=16", spec_8b, 10, 512, 64, 16),
        "8b_98x512": make_workload("8B long: 98x512 + 64 query, k=16", spec_8b, 98, 512, 64, 16),
        "8b_32req": make_workload("8B batched: 32 req x (8x512 Zipf from 64) + 32 query, k=16",
                            spec_8b, 64, 512, 32, 16, n_requests=32, pool=64, per_request=8),
    }
    for k in (0, 2, 16, 32, 512):
        w[f"8b_10x512_k{k}"] = make_workload(f"8B ablation: 10x512 + 64 query, k={k}", spec_8b, 10, 512, 64, k,
                                      n_dummy=N_DUMMY_LEGOLINK0 if k == 0 else 0)
    return w
