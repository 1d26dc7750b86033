"""Parity of the link step at the evaluated configurations (Llama-3-8B shape, bf16).

Every case runs the library at the configuration's full size (32 layers, 512-token
chunks) and compares with the fp64 oracle on outputs the oracle can compute exactly in
bounded time. Compiled chunk KV is a seeded stand-in imported into both stores (the
link's arithmetic does not depend on how the chunk KV was produced; compile itself is
checked at the same width with fewer layers).

  10 x 512 + 64 query, k in {0, 2, 16, 32}: every output, 32 layers; at k = 16
      also one decode step after the link (hidden, logits, the new K/V row of every layer).
  10 x 512 + 64, k = 512 (full recompute): recomputed K/V of chunks 1-2 at every layer (they depend
      only on those chunks), compared with a plain prefill of chunks 1-2.
  98 x 512 + 64, k = 16: recomputed K/V of the first 4 chunks' rows at every layer
      (prefix sample), plus a 2-layer model over the whole 50k-token prompt, every output.
  98 x 512 + 64 also against stored fp64 oracle outputs of the whole 32-layer link (the 64 query rows'
      hidden states, the last row's logits, sampled recomputed K/V rows at sampled layers),
      written by tests/golden/make_long_98x512_golden.py.
  32 requests x 8 Zipf chunks + 32 query: requests 1, 2, 16 and 32 (the last) in full,
      out of the batch of 32.
Page tables, slots and selected lists are compared bit-exactly for every request.
"""
import os

import numpy as np
import pytest
import torch

import pic_inputs as pi
from oracle import pic_oracle as po
from tests.helpers import rel_err

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def m8b():
    from position_independent_kv_link_gb300 import PicModel
    spec = pi.LLAMA3_8B
    w = pi.gen_weights(spec)
    model = PicModel(spec, w)
    yield spec, w, model, po.OracleModel(spec, w)
    model.close()


def _store(model, wl, extra_blocks=2048, rows=None):
    from position_independent_kv_link_gb300 import PicStore
    n_pos = max(sum(len(wl.chunks[c]) for c in r.chunk_ids) + len(r.query) for r in wl.requests)
    nb = sum(-(-len(c) // 16) for c in wl.chunks) + extra_blocks
    return PicStore(model, num_blocks=nb, max_rows=max(rows or wl.selected_rows, 256),
                    max_requests=max(64, len(wl.requests)), max_positions=n_pos + 16,
                    max_logit_rows=max(64, len(wl.requests)))


def _import(store, spec, wl, chunk_ids, ost=None):
    """Seeded stand-in KV of the listed chunks, imported into the library (and oracle) store."""
    g, o = {}, {}
    for c in chunk_ids:
        k, v = pi.gen_chunk_kv(spec, len(wl.chunks[c]), c)
        g[c] = store.import_chunk(wl.chunks[c], k.cuda(), v.cuda())
        if ost is not None:
            o[c] = ost.import_chunk(wl.chunks[c], [k[l] for l in range(spec.n_layers)],
                                    [v[l] for l in range(spec.n_layers)])
    return g, o


def _meta_oracle(wl, order, requests):
    """The oracle's integer metadata for `requests` after importing chunks in `order`."""
    st = po.OracleStore(None, 1 << 16)
    ids = {c: st._add_chunk(np.asarray(wl.chunks[c]), [], []) for c in order}
    return st.plan([([ids[c] for c in r.chunk_ids], len(r.query)) for r in requests], wl.k)


def _check_meta(store, handles, metas):
    for h, m in zip(handles, metas):
        info = store.request_info(h)
        for key in ("selected", "slots", "page_table", "page_pos", "page_len", "private_blocks"):
            assert np.array_equal(info[key], getattr(m, key)), key


def _check_kv(store, handle, ref_k, ref_v, layers, rows=None):
    info = store.request_info(handle)
    slots = info["slots"] if rows is None else info["slots"][rows]
    worst = 0.0
    for l in layers:
        k, v = store.kv_rows(l, slots)
        worst = max(worst, rel_err(k, ref_k[l]), rel_err(v, ref_v[l]))
    assert worst <= TOL, worst
    return worst


# ----------------------------------------------------------------------------- 10 x 512 + 64 and the k sweep

@pytest.mark.parametrize("k", [16, 0, 2, 32])
def test_10x512_k_sweep_full_outputs(m8b, k):
    spec, w, model, om = m8b
    wl = pi.config_workloads()[f"8b_10x512_k{k}"]
    store = _store(model, wl)
    ost = po.OracleStore(om, 1 << 14)
    order = list(range(len(wl.chunks)))
    g, o = _import(store, spec, wl, order, ost)
    r = wl.requests[0]
    res = store.link([([g[c] for c in r.chunk_ids], r.query)], wl.k)
    store.sync()
    _check_meta(store, res.requests, _meta_oracle(wl, order, wl.requests))
    out = ost.link([([o[c] for c in r.chunk_ids], r.query)], wl.k)
    assert rel_err(res.hidden, out.hidden[0]) <= TOL
    assert rel_err(res.logits, out.logits[0]) <= TOL
    _check_kv(store, res.requests[0], out.k[0], out.v[0], range(spec.n_layers))
    if k == 16:   # one decode step after the link, at the size the benchmark times it
        tok = [int(pi.gen_tokens(1, spec.vocab, 63)[0])]
        d = store.decode(res.requests, tok)
        store.sync()
        od = ost.decode(out.rids, tok)
        assert d.positions.tolist() == od.positions.tolist() and d.slots.tolist() == od.slots.tolist()
        assert rel_err(d.hidden, od.hidden) <= TOL and rel_err(d.logits, od.logits) <= TOL
        for l in range(spec.n_layers):
            kk, vv = store.kv_rows(l, d.slots)
            assert rel_err(kk, od.k[0][l][None]) <= TOL and rel_err(vv, od.v[0][l][None]) <= TOL
    store.close()


def test_10x512_full_recompute_prefix(m8b):
    """k = 512 recomputes every row; rows of chunks 1-2 equal a plain prefill of those chunks."""
    spec, w, model, om = m8b
    wl = pi.config_workloads()["8b_10x512_k512"]
    store = _store(model, wl)
    order = list(range(len(wl.chunks)))
    g, _ = _import(store, spec, wl, order)
    r = wl.requests[0]
    res = store.link([([g[c] for c in r.chunk_ids], r.query)], wl.k)
    store.sync()
    _check_meta(store, res.requests, _meta_oracle(wl, order, wl.requests))
    fr = po.full_prefill(om, np.concatenate([wl.chunks[0], wl.chunks[1]]))
    _check_kv(store, res.requests[0], fr.k, fr.v, range(spec.n_layers), rows=slice(0, 1024))
    store.close()


# ----------------------------------------------------------------------------- 98 x 512 + 64 (long context)

LONG_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "long_98x512_link_outputs.npz")


def test_98x512_all_layers(m8b):
    """The 98-chunk, 50k-token link through all 32 layers. (1) The 64 query rows' final hidden
    states, the last row's logits and sampled recomputed K/V rows against the fp64 oracle's
    outputs, computed once by tests/golden/make_long_98x512_golden.py from the same seeded weights and
    chunk KV. (2) The recomputed K/V of the first 4 chunks' rows at every layer against an
    oracle link of those chunks (they depend on nothing later)."""
    spec, w, model, om = m8b
    wl = pi.config_workloads()["8b_98x512"]
    store = _store(model, wl)
    order = list(range(len(wl.chunks)))
    g, _ = _import(store, spec, wl, order)
    r = wl.requests[0]
    res = store.link([([g[c] for c in r.chunk_ids], r.query)], wl.k)
    store.sync()
    _check_meta(store, res.requests, _meta_oracle(wl, order, wl.requests))
    gold = np.load(LONG_GOLDEN)
    info = store.request_info(res.requests[0])
    assert np.array_equal(info["selected"], gold["selected"])
    assert rel_err(res.hidden, gold["hidden"]) <= TOL
    assert rel_err(res.logits, gold["logits"]) <= TOL
    slots = info["slots"][gold["kv_rows"]]
    for i, l in enumerate(gold["kv_layers"]):
        k, v = store.kv_rows(int(l), slots)
        assert rel_err(k, gold["k"][i]) <= TOL and rel_err(v, gold["v"][i]) <= TOL, int(l)
    # rows of chunks 1-4 depend on those chunks only: an oracle link over them gives their KV
    ost = po.OracleStore(om, 1 << 12)
    _, o = _import(_NullStore(), spec, wl, range(4), ost)
    out = ost.link([([o[c] for c in range(4)], r.query)], wl.k)
    n = 4 * wl.k
    _check_kv(store, res.requests[0], [a[:n] for a in out.k[0]], [a[:n] for a in out.v[0]], range(spec.n_layers),
              rows=slice(0, n))
    store.close()


class _NullStore:
    def import_chunk(self, *a, **k):
        return None


def test_98x512_two_layer_full_outputs():
    """The whole 50k-token, 98-chunk link with a 2-layer model of the same width: every output."""
    from position_independent_kv_link_gb300 import PicModel
    spec = pi.LLAMA3_8B.with_layers(2)
    w = pi.gen_weights(spec)
    model = PicModel(spec, w)
    om = po.OracleModel(spec, w)
    wl = pi.config_workloads(spec)["8b_98x512"]
    store = _store(model, wl)
    ost = po.OracleStore(om, 1 << 13)
    g, o = _import(store, spec, wl, range(len(wl.chunks)), ost)
    r = wl.requests[0]
    res = store.link([([g[c] for c in r.chunk_ids], r.query)], wl.k)
    store.sync()
    out = ost.link([([o[c] for c in r.chunk_ids], r.query)], wl.k)
    assert rel_err(res.hidden, out.hidden[0]) <= TOL
    assert rel_err(res.logits, out.logits[0]) <= TOL
    _check_kv(store, res.requests[0], out.k[0], out.v[0], range(spec.n_layers))
    store.close()
    model.close()


# ----------------------------------------------------------------------------- 32 requests (batched, shared pool)

def test_32req_batched_sampled_requests(m8b):
    spec, w, model, om = m8b
    wl = pi.config_workloads()["8b_32req"]
    store = _store(model, wl)
    order = sorted({c for r in wl.requests for c in r.chunk_ids})
    g, _ = _import(store, spec, wl, order)
    res = store.link([([g[c] for c in r.chunk_ids], r.query) for r in wl.requests], wl.k)
    store.sync()
    _check_meta(store, res.requests, _meta_oracle(wl, order, wl.requests))
    sample = [0, 1, 15, 31]
    need = sorted({c for i in sample for c in wl.requests[i].chunk_ids})
    ost = po.OracleStore(om, 1 << 13)
    _, o = _import(_NullStore(), spec, wl, need, ost)
    out = ost.link([([o[c] for c in wl.requests[i].chunk_ids], wl.requests[i].query) for i in sample], wl.k)
    lq = len(wl.requests[0].query)
    for j, i in enumerate(sample):
        assert rel_err(res.hidden[i * lq:(i + 1) * lq], out.hidden[j]) <= TOL
        assert rel_err(res.logits[i:i + 1], out.logits[j]) <= TOL
        _check_kv(store, res.requests[i], out.k[j], out.v[j], range(spec.n_layers))
    store.close()


# ----------------------------------------------------------------------------- compile at the 8B width

@pytest.mark.parametrize("n_dummy,k", [(0, 16), (4, 0)])
def test_compile_then_link_8b_width(n_dummy, k):
    """pic_compile at the 8B width (2 layers, 3 x 512 chunks), LegoLink-0 dummies included."""
    from position_independent_kv_link_gb300 import PicModel
    from tests.helpers import compare_link, library_run, oracle_run
    spec = pi.LLAMA3_8B.with_layers(2)
    w = pi.gen_weights(spec)
    model = PicModel(spec, w)
    wl = pi.make_workload("8B-width compile", spec, 3, 512, 64, k, n_dummy=n_dummy)
    store = _store(model, wl, rows=2048)
    _, res = library_run(store, wl)
    _, _, out = oracle_run(po.OracleModel(spec, w), wl, 1 << 12)
    compare_link(store, res, out, spec)
    store.close()
    model.close()
