"""Content-addressed chunk reuse and LRU eviction in the paged store (pic_compile_cached).

A chunk is compiled once and linked into any prompt; the store keeps one shared copy of its
KV for every request that uses it. These tests follow block ids by hand on the tiny fp32
model (64-token chunks = 4 blocks): reuse returns the resident chunk without new blocks,
released cached chunks stay resident until evicted least recently released first, eviction
happens only when it lets a call succeed, and links over reused or re-compiled chunks match
the fp64 oracle (outputs within 1e-4, page tables bit-exact).
"""
import numpy as np
import pytest
import torch

import pic_inputs as pi
from oracle import pic_oracle as po
from tests.helpers import compare_link, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def tiny():
    from position_independent_kv_link_gb300 import PicModel
    spec = pi.TINY
    w = pi.gen_weights(spec, gains="random")
    return spec, w, PicModel(spec, w), po.OracleModel(spec, w)


def _store(model, nb):
    from position_independent_kv_link_gb300 import PicStore
    return PicStore(model, num_blocks=nb, max_rows=2048, max_requests=16, max_positions=8192, max_logit_rows=64)


def _chunk(spec, i, n=64):
    return pi.gen_tokens(n, spec.vocab, 70, i)


def test_reuse_returns_resident_chunks_and_links_like_the_oracle(tiny):
    spec, w, model, om = tiny
    wl = pi.config_workloads()["tiny"]                  # 4 x 64 + 16 query, k = 2
    store = _store(model, 64)
    ids, hits = store.compile_cached(wl.chunks)
    assert hits == [False] * 4 and store.free_blocks() == 64 - 16
    ids2, hits2 = store.compile_cached(wl.chunks)
    assert ids2 == ids and hits2 == [True] * 4 and store.free_blocks() == 64 - 16
    st = store.cache_stats()
    assert (st["hits"], st["misses"], st["cached_chunks"], st["unreferenced_chunks"]) == (4, 4, 4, 0)
    r = wl.requests[0]
    res = store.link([([ids[c] for c in r.chunk_ids], r.query)], wl.k)
    store.sync()
    _, _, out = oracle_run(om, wl, 64)                   # same lowest-free block ids
    compare_link(store, res, out, spec)


def test_identical_chunks_in_one_call_compile_once(tiny):
    spec, w, model, om = tiny
    store = _store(model, 64)
    A, B = _chunk(spec, 0), _chunk(spec, 1)
    ids, hits = store.compile_cached([A, A, B])
    assert ids[0] == ids[1] != ids[2] and hits == [False, True, False]
    assert store.free_blocks() == 64 - 8
    store.release_chunk(ids[0])
    assert store.cache_stats()["unreferenced_chunks"] == 0    # the second reference holds it
    store.release_chunk(ids[1])
    store.release_chunk(ids[2])
    st = store.cache_stats()
    assert st["unreferenced_chunks"] == 2 and st["unreferenced_blocks"] == 8 and store.free_blocks() == 56
    assert store.evict() == 2 and store.free_blocks() == 64 and store.cache_stats()["evictions"] == 2


def test_lru_eviction_order_and_all_or_nothing(tiny):
    from position_independent_kv_link_gb300 import PicError
    from position_independent_kv_link_gb300 import _lib as L
    spec, w, model, om = tiny
    store = _store(model, 12)                            # room for three 4-block chunks
    A, B, C, D = (_chunk(spec, i) for i in range(4))
    (a,), _ = store.compile_cached([A])                  # blocks 0-3
    (b,), _ = store.compile_cached([B])                  # 4-7
    (c,), _ = store.compile_cached([C])                  # 8-11
    assert store.free_blocks() == 0
    store.release_chunk(a)
    store.release_chunk(b)                               # unreferenced, released in the order a, b
    st = store.cache_stats()
    assert (st["unreferenced_chunks"], st["unreferenced_blocks"], st["blocks_in_use"]) == (2, 8, 12)
    (d,), (hit,) = store.compile_cached([D])             # evicts a (released first) and takes 0-3
    assert not hit and store.chunk_blocks(d).tolist() == [0, 1, 2, 3] and store.cache_stats()["evictions"] == 1
    (b2,), (hit,) = store.compile_cached([B])            # b is still resident
    assert hit and b2 == b and store.chunk_blocks(b).tolist() == [4, 5, 6, 7]
    before = store.cache_stats()
    with pytest.raises(PicError) as e:                   # a was evicted; b, c, d are referenced
        store.compile_cached([A])
    assert e.value.status == L.PIC_ERR_OUT_OF_BLOCKS
    assert store.cache_stats() == before and store.free_blocks() == 0
    store.release_chunk(d)
    (a2,), (hit,) = store.compile_cached([A])            # evicts d, recompiles A into 0-3
    assert not hit and a2 not in (a, d) and store.chunk_blocks(a2).tolist() == [0, 1, 2, 3]
    # a link that needs blocks evicts too: release c, link [A, B] + query (2 private + 1 query)
    store.release_chunk(c)
    q = pi.gen_tokens(16, spec.vocab, 71)
    res = store.link([([a2, b], q)], 2)
    store.sync()
    st = store.cache_stats()
    assert st["evictions"] == 3 and st["hits"] == 1 and st["misses"] == 5
    wl = pi.Workload("lru", spec, [A, B], [pi.Request([0, 1], q)], 2, 0)
    _, _, out = oracle_run(om, wl, 12)                   # A 0-3, B 4-7, privates 8, 9, query 10
    compare_link(store, res, out, spec)


def test_released_cached_handles_are_invalid_and_requests_hold_chunks(tiny):
    from position_independent_kv_link_gb300 import PicError
    from position_independent_kv_link_gb300 import _lib as L
    spec, w, model, om = tiny
    store = _store(model, 32)
    A = _chunk(spec, 5)
    (a,), _ = store.compile_cached([A])
    res = store.link([([a], pi.gen_tokens(8, spec.vocab, 72))], 2)
    store.sync()
    store.release_chunk(a)                               # the request still references it
    assert store.cache_stats()["unreferenced_chunks"] == 0
    store.release_request(res.requests[0])
    assert store.cache_stats()["unreferenced_chunks"] == 1
    for call in (lambda: store.release_chunk(a), lambda: store.chunk_blocks(a),
                 lambda: store.link([([a], np.zeros(4, dtype=np.int32))], 2)):
        with pytest.raises(PicError) as e:
            call()
        assert e.value.status == L.PIC_ERR_INVALID_ARG
    (a2,), (hit,) = store.compile_cached([A])
    assert hit and a2 == a and store.cache_stats()["unreferenced_chunks"] == 0
    # chunks from the plain compile are not cached: their blocks return at their last release
    (p,) = store.compile([A])
    free = store.free_blocks()
    store.release_chunk(p)
    assert store.free_blocks() == free + 4 and store.cache_stats()["cached_chunks"] == 1


def test_kv_hbm_in_use_with_shared_chunks(tiny):
    """Paged sharing (MEPIC): a pool of 6 chunks linked by 4 requests of 3 chunks each, k = 2,
    holds each chunk once plus one private block per chunk per request and the query pages."""
    spec, w, model, om = tiny
    store = _store(model, 128)
    pool = [_chunk(spec, 10 + i) for i in range(6)]
    ids, _ = store.compile_cached(pool)
    picks = [[0, 1, 2], [3, 4, 5], [0, 2, 4], [1, 3, 5]]
    queries = [pi.gen_tokens(16, spec.vocab, 73, r) for r in range(4)]
    store.link([([ids[c] for c in p], q) for p, q in zip(picks, queries)], 2)
    store.sync()
    st = store.cache_stats()
    shared = 6 * 4 + 4 * (3 * 1 + 1)                    # chunk pages once + privates + query pages
    unshared = 4 * (3 * 4 + 1)                           # every request holding its own prompt
    assert st["blocks_in_use"] == shared
    assert st["block_bytes"] == 2 * spec.n_layers * spec.n_kv_heads * 16 * spec.head_dim * 4
    assert shared < unshared
