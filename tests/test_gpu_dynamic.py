"""GPU parity of dynamic (attention-based) token selection, pic_link_dynamic, against the oracle.

The reading (the CacheBlend-r step of the EPIC pages): each prompt token scores the layer-0
softmax mass the query rows put on it, with nothing recomputed; the floor(r N / 100) best
are recomputed, equal scores taken in position order. Checked here:

  * the scores (fp32 on the GPU) against the oracle's fp64 scores, within the tolerance of
    the model dtype;
  * the chosen positions: exactly the oracle's rule (select_top) applied to the GPU's own
    fp32 scores -- the integer decision taken in the kernel's precision -- and the oracle's
    own choice on its fp64 scores for every token further than twice the largest score
    deviation from the threshold score;
  * exact ties (a prompt whose compiled K is zero gets identical scores everywhere): the
    first n positions;
  * page tables, slots, selected lists and private blocks bit-exact against the oracle's
    plan over the GPU's choice, and hidden states, logits and every recomputed K/V row of
    the link within tolerance;
  * r = 0 (naive reuse) and r = 100 (full recompute) against pic_link with k = 0 and with
    k = the longest chunk;
  * the 8B shape at full size (10 x 512 + 64 query): scores, choice and metadata, and the
    whole 32-layer link at r = 10.
"""
import numpy as np
import pytest
import torch

import pic_inputs as pi
from oracle import pic_oracle as po
from tests.helpers import compare_link, rel_err, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    from position_independent_kv_link_gb300 import load
    load()


def _stores(spec, w, n_blocks=512, rows=1024, positions=4096):
    from position_independent_kv_link_gb300 import PicModel, PicStore
    model = PicModel(spec, w)
    store = PicStore(model, num_blocks=n_blocks, max_rows=rows, max_requests=8, max_positions=positions,
                     max_logit_rows=256)
    return model, store


def _check_choice(info_sel, n_prompt, lq, scores_gpu, scores_or, r, tol):
    """The request's chosen prompt positions (its selected list minus the query rows)."""
    chosen = np.asarray(info_sel[:len(info_sel) - lq], dtype=np.int64)
    assert np.array_equal(np.asarray(info_sel[len(info_sel) - lq:]), np.arange(n_prompt, n_prompt + lq))
    n = r * n_prompt // 100
    assert len(chosen) == n
    # the oracle's rule on the GPU's fp32 scores: the same integer decision, bit-exact
    assert np.array_equal(chosen, po.select_top(np.asarray(scores_gpu, dtype=np.float64), r))
    # the oracle's choice on its own fp64 scores, away from the threshold: with e the largest
    # score deviation, the n-th largest GPU score is within e of the oracle's, so a token more
    # than 2e above (below) the oracle's threshold is (is not) chosen whatever the rounding
    assert rel_err(scores_gpu, scores_or) <= tol
    if 0 < n < n_prompt:
        e = float(np.max(np.abs(np.asarray(scores_gpu, dtype=np.float64) - scores_or)))
        thr = np.sort(scores_or)[::-1][n - 1]
        must = np.nonzero(scores_or > thr + 2 * e)[0]
        never = np.nonzero(scores_or < thr - 2 * e)[0]
        assert set(must.tolist()) <= set(chosen.tolist())
        assert not set(never.tolist()) & set(chosen.tolist())
    return chosen


def _split(chosen, lens):
    """Prompt positions -> per chunk local indices."""
    out, off = [], 0
    for L in lens:
        out.append([int(u - off) for u in chosen if off <= u < off + L])
        off += L
    return out


def _run(spec, wl, rs):
    """pic_link_dynamic for each r (one store, requests released in between) against the oracle."""
    w = pi.gen_weights(spec)
    om = po.OracleModel(spec, w)
    model, store = _stores(spec, w)
    tol = tol_for(spec)
    try:
        cids = store.compile(wl.chunks, n_dummy=wl.n_dummy)
        ost = po.OracleStore(om, 512)
        ocids = ost.compile_many(wl.chunks, wl.n_dummy)
        reqs = [([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests]
        oreqs = [([ocids[c] for c in r.chunk_ids], r.query) for r in wl.requests]
        for r in rs:
            n_tok = sum(len(wl.chunks[c]) for q in wl.requests for c in q.chunk_ids)
            scores = torch.full((n_tok,), -1.0, dtype=torch.float32, device="cuda")
            res = store.link_dynamic(reqs, r, all_logits=True, scores_out=scores)
            store.sync()
            sc = scores.cpu().double().numpy()
            sels, off = [], 0
            for i, q in enumerate(wl.requests):
                lens = [len(wl.chunks[c]) for c in q.chunk_ids]
                N = sum(lens)
                chs = [ost.chunks[ocids[c]] for c in q.chunk_ids]
                so = po.query_attention_scores(om, [c.tokens for c in chs], [c.k[0] for c in chs], q.query)
                info = store.request_info(res.requests[i])
                chosen = _check_choice(info["selected"], N, len(q.query), sc[off:off + N], so, r, tol)
                sels.append(_split(chosen, lens))
                off += N
            out = ost.link_selected([(c, q, s) for (c, q), s in zip(oreqs, sels)], all_logits=True)
            compare_link(store, res, out, spec)
            for h in res.requests:
                store.release_request(h)
            for rid in list(ost.requests):
                ost.release_request(rid)
            assert store.free_blocks() == len(ost.free)
    finally:
        store.close()
        model.close()


def test_tiny_f32_dynamic():
    wl = pi.config_workloads()["tiny"]
    _run(pi.TINY, wl, [10, 25, 50, 0, 100])


def test_small_bf16_dynamic_batch_of_three():
    """Three requests, ragged chunks, one chunk in two requests, chunk orders differ."""
    spec = pi.SMALL_BF16
    wl = pi.make_workload("dyn bf16", spec, 5, [64, 40, 100, 17, 33], 24, 0, n_requests=3, pool=5, per_request=3)
    _run(spec, wl, [20, 7])


def test_r0_and_r100_match_static_link():
    """r = 0: the query alone (pic_link, k = 0); r = 100: every token (k = longest chunk). Same
    metadata as pic_link, and the same outputs as the oracle's static link."""
    spec = pi.SMALL_BF16
    wl = pi.make_workload("dyn ends", spec, 3, [48, 20, 37], 16, 0)
    w = pi.gen_weights(spec)
    om = po.OracleModel(spec, w)
    model, store = _stores(spec, w)
    try:
        cids = store.compile(wl.chunks)
        reqs = [([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests]
        for r, k in ((0, 0), (100, 48)):
            a = store.link_dynamic(reqs, r, all_logits=True)
            store.sync()
            ia = store.request_info(a.requests[0])
            ost = po.OracleStore(om, 512)
            ocids = ost.compile_many(wl.chunks)
            out = ost.link([([ocids[c] for c in q.chunk_ids], q.query) for q in wl.requests], k, all_logits=True)
            compare_link(store, a, out, spec)
            store.release_request(a.requests[0])
            b = store.link(reqs, k, all_logits=True)
            store.sync()
            ib = store.request_info(b.requests[0])
            for key in ia:
                assert np.array_equal(ia[key], ib[key]), (r, key)
            store.release_request(b.requests[0])
    finally:
        store.close()
        model.close()


def test_exact_ties_take_the_first_positions():
    """Zero compiled K: every prompt token's logit is 0, so all scores are equal; the top n are
    positions 0..n-1 (the tie rule), on the GPU and in the oracle."""
    spec = pi.SMALL_BF16
    wl = pi.make_workload("dyn ties", spec, 3, [40, 64, 23], 16, 0)
    w = pi.gen_weights(spec)
    om = po.OracleModel(spec, w)
    model, store = _stores(spec, w)
    try:
        hs, os_ = [], []
        ost = po.OracleStore(om, 512)
        for i, c in enumerate(wl.chunks):
            k, v = pi.gen_chunk_kv(spec, len(c), i)
            k = torch.zeros_like(k)
            hs.append(store.import_chunk(c, k.cuda(), v.cuda()))
            os_.append(ost.import_chunk(c, [k[l] for l in range(spec.n_layers)], [v[l] for l in range(spec.n_layers)]))
        q = wl.requests[0].query
        N = sum(len(c) for c in wl.chunks)
        scores = torch.empty(N, dtype=torch.float32, device="cuda")
        res = store.link_dynamic([(hs, q)], 30, scores_out=scores)
        store.sync()
        sc = scores.cpu().numpy()
        assert np.all(sc == sc[0])
        n = 30 * N // 100
        info = store.request_info(res.requests[0])
        assert np.array_equal(info["selected"][:n], np.arange(n))
        out, (so,) = ost.link_dynamic([(os_, q)], 30)
        assert np.all(so == so[0])
        for key in ("selected", "slots", "page_table", "page_pos", "page_len", "private_blocks"):
            assert np.array_equal(info[key], getattr(out.meta[0], key)), key
        assert rel_err(res.hidden, out.hidden[0]) <= 2e-2
        assert rel_err(res.logits, out.logits[0]) <= 2e-2
    finally:
        store.close()
        model.close()


def test_8b_shape_dynamic_full_size():
    """10 x 512 + 64 query at the 8B shape (seeded stand-in chunk KV in both stores): scores and
    choice at r = 15 and r = 10, metadata, and the whole 32-layer link at r = 10."""
    from position_independent_kv_link_gb300 import PicModel, PicStore
    spec = pi.LLAMA3_8B
    wl = pi.config_workloads()["8b_10x512"]
    w = pi.gen_weights(spec)
    om = po.OracleModel(spec, w)
    model = PicModel(spec, w)
    store = PicStore(model, num_blocks=2048, max_rows=1024, max_requests=8, max_positions=5248, max_logit_rows=64)
    try:
        ost = po.OracleStore(om, 1 << 14)
        g, o = [], []
        for c, toks in enumerate(wl.chunks):
            k, v = pi.gen_chunk_kv(spec, len(toks), c)
            g.append(store.import_chunk(toks, k.cuda(), v.cuda()))
            o.append(ost.import_chunk(toks, [k[l] for l in range(spec.n_layers)], [v[l] for l in range(spec.n_layers)]))
        q = wl.requests[0].query
        lens = [len(c) for c in wl.chunks]
        N = sum(lens)
        chs = [ost.chunks[c] for c in o]
        so = po.query_attention_scores(om, [c.tokens for c in chs], [c.k[0] for c in chs], q)
        for r in (15, 10):
            scores = torch.empty(N, dtype=torch.float32, device="cuda")
            res = store.link_dynamic([(g, q)], r, scores_out=scores)
            store.sync()
            info = store.request_info(res.requests[0])
            chosen = _check_choice(info["selected"], N, len(q), scores.cpu().double().numpy(), so, r, 2e-2)
            if r == 10:
                out = ost.link_selected([(o, q, _split(chosen, lens))])
                compare_link(store, res, out, spec)
                ost.release_request(next(iter(ost.requests)))
            else:
                meta = ost.plan_selected([(o, len(q), _split(chosen, lens))])[0]
                for key in ("selected", "slots", "page_table", "page_pos", "page_len", "private_blocks"):
                    assert np.array_equal(info[key], getattr(meta, key)), key
                ost.free.update(meta.private_blocks.tolist())
            store.release_request(res.requests[0])
    finally:
        store.close()
        model.close()
