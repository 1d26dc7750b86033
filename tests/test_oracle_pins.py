"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

* RoPE: closed forms (composition, relative position, norm, identity at 0) and a
  complex-multiplication formulation.
* RMSNorm and the whole prefill: torch library routines (rms_norm,
  scaled_dot_product_attention, complex RoPE) in float64.
* Link: the special cases the method reduces to (k = chunk length is full recompute;
  a single chunk with k = 0 is a plain prefill), chunk 1 reproduces its compile,
  compile is offset invariant, and a brute-force per-token loop agrees.
* Decode after link: with k = chunk length (and for one chunk with k = 0) each decoded
  token continues a plain prefill; otherwise it agrees with the brute-force twin, which
  generates from its own link's caches; page growth follows a hand-worked example.
* Metadata: a hand-worked example and closed forms.
* Planted mistakes: each pin is shown to fail when the oracle is broken on purpose.
"""
import json
import os

import numpy as np
import pytest
import torch

import pic_inputs as pi
from oracle import pic_oracle as po
from oracle import bruteforce as bf
from tests import torch_reference as tr

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _weights(spec, gains="random"):
    return pi.gen_weights(spec, gains=gains)


@pytest.fixture(scope="module")
def micro():
    w = _weights(pi.MICRO_GQA)
    return pi.MICRO_GQA, w, po.OracleModel(pi.MICRO_GQA, w)


@pytest.fixture(scope="module")
def tiny():
    w = _weights(pi.TINY)
    return pi.TINY, w, po.OracleModel(pi.TINY, w)


def rel_err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b))))


# ----------------------------------------------------------------------------- RoPE

def test_rope_composition_relative_norm():
    rng = np.random.default_rng(0)
    D, base = 128, 500000.0
    x = rng.standard_normal((7, 3, D))
    p = np.array([0, 1, 5, 100, 4096, 50000, 50239])
    d = np.array([3, 0, 17, 511, 9, 1, 2])
    # R(d) R(p) = R(p + d)
    assert np.allclose(po.rope(po.rope(x, p, base), d, base), po.rope(x, p + d, base), atol=1e-9)
    # R(0) is the identity
    assert np.array_equal(po.rope(x, np.zeros(7, dtype=int), base), x)
    # |R(p) x| = |x|
    assert np.allclose(np.linalg.norm(po.rope(x, p, base), axis=-1), np.linalg.norm(x, axis=-1))
    # <R(p) q, R(p') k> depends only on p - p'
    q, k = rng.standard_normal((1, 1, D)), rng.standard_normal((1, 1, D))
    def dot(a, b):
        return float(np.sum(po.rope(q, np.array([a]), base) * po.rope(k, np.array([b]), base)))
    assert abs(dot(10, 3) - dot(1010, 1003)) < 1e-9
    assert abs(dot(40000, 123) - dot(39877, 0)) < 1e-8


def test_rope_matches_complex_multiplication():
    rng = np.random.default_rng(1)
    for D, base in ((64, 10000.0), (128, 500000.0), (16, 10000.0)):
        x = rng.standard_normal((9, 2, D))
        pos = np.array([0, 1, 2, 15, 16, 511, 512, 5183, 50239])
        ref = tr.complex_rope(torch.from_numpy(x), torch.from_numpy(pos), base).numpy()
        # angles up to 5e4 rad carry ~pos * 1e-16 rounding in fp64
        assert rel_err(po.rope(x, pos, base), ref) < 1e-10


def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 256)) * 3
    g = rng.standard_normal(256)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (256,), torch.from_numpy(g), 1e-5).numpy()
    assert rel_err(po.rms_norm(x, g, 1e-5), ref) < 1e-14
    # closed form: a constant row c maps to c/sqrt(c^2+eps) * g
    c = np.full((1, 8), 2.0)
    assert np.allclose(po.rms_norm(c, np.ones(8), 0.0), np.ones((1, 8)))


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((6, 4, 16))
    k = rng.standard_normal((9, 2, 16))
    v = np.ones((9, 2, 16))
    qp, kp = np.array([0, 2, 3, 5, 7, 8]), np.arange(9)
    assert np.allclose(po.causal_attention(q, k, v, qp, kp), 1.0)
    # a row that sees only itself returns that row's value
    v2 = rng.standard_normal((9, 2, 16))
    out = po.causal_attention(q, k, v2, qp, kp)
    assert np.allclose(out[0, 0], v2[0, 0]) and np.allclose(out[0, 3], v2[0, 1])


# ----------------------------------------------------------------------------- whole model vs library routines

@pytest.mark.parametrize("name", ["micro", "tiny"])
def test_prefill_matches_torch_library(name, micro, tiny):
    spec, w, model = {"micro": micro, "tiny": tiny}[name]
    toks = pi.gen_tokens(37 if name == "micro" else 80, spec.vocab, 99, name)
    got = po.full_prefill(model, toks)
    hid, logits, ks, vs = tr.prefill(spec, w, toks)
    assert rel_err(got.hidden, hid.numpy()) < 1e-11
    assert rel_err(model.logits(got.hidden[-1:]), logits.numpy()) < 1e-11
    for l in range(spec.n_layers):
        assert rel_err(got.k[l], ks[l].numpy()) < 1e-11
        assert rel_err(got.v[l], vs[l].numpy()) < 1e-11


# ----------------------------------------------------------------------------- link special cases

def _link(spec, model, chunks, queries, k, n_dummy=0, num_blocks=256, all_logits=False):
    st = po.OracleStore(model, num_blocks)
    cids = st.compile_many(chunks, n_dummy)
    out = st.link([(cids, q) for q in queries], k, all_logits=all_logits)
    return st, cids, out


def test_full_recompute_invariant(tiny, micro):
    """k >= every chunk length: link equals a plain prefill of the concatenated prompt."""
    for spec, w, model in (tiny, micro):
        lens = [64, 64, 64, 64] if spec is pi.TINY else [5, 16, 19]
        chunks = [pi.gen_tokens(L, spec.vocab, 7, i) for i, L in enumerate(lens)]
        q = pi.gen_tokens(16 if spec is pi.TINY else 6, spec.vocab, 8)
        _, _, out = _link(spec, model, chunks, [q], k=max(lens), all_logits=True)
        fr = po.full_prefill(model, np.concatenate(chunks + [q]))
        assert rel_err(out.hidden[0], fr.hidden[-len(q):]) < 1e-11
        assert rel_err(out.logits[0], model.logits(fr.hidden[-len(q):])) < 1e-11
        for l in range(spec.n_layers):
            assert rel_err(out.k[0][l], fr.k[l]) < 1e-11
            assert rel_err(out.v[0][l], fr.v[l]) < 1e-11


def test_single_chunk_k0_is_plain_prefill(tiny):
    spec, w, model = tiny
    chunk = pi.gen_tokens(64, spec.vocab, 11)
    q = pi.gen_tokens(16, spec.vocab, 12)
    _, _, out = _link(spec, model, [chunk], [q], k=0)
    fr = po.full_prefill(model, np.concatenate([chunk, q]))
    assert rel_err(out.hidden[0], fr.hidden[-16:]) < 1e-11
    assert rel_err(out.logits[0], model.logits(fr.hidden[-1:])) < 1e-11


def test_chunk1_recompute_equals_compile(tiny):
    spec, w, model = tiny
    chunks = [pi.gen_tokens(64, spec.vocab, 13, i) for i in range(3)]
    q = pi.gen_tokens(16, spec.vocab, 14)
    st, cids, out = _link(spec, model, chunks, [q], k=2)
    for l in range(spec.n_layers):
        assert rel_err(out.k[0][l][:2], st.chunks[cids[0]].k[l][:2]) < 1e-11
        assert rel_err(out.v[0][l][:2], st.chunks[cids[0]].v[l][:2]) < 1e-11
        # layer 0 K/V depend on the token alone; deeper layers of later chunks change
        # once their first rows see the prefix
        d = rel_err(out.k[0][l][2:4], st.chunks[cids[1]].k[l][:2])
        assert (d < 1e-12) if l == 0 else (d > 1e-6)


def test_compile_offset_invariance(tiny):
    """Pre-RoPE KV of an isolated chunk does not depend on where its positions start."""
    spec, w, model = tiny
    chunk = pi.gen_tokens(40, spec.vocab, 15)
    ref = po.full_prefill(model, chunk)
    for delta in (1, 517, 20000):
        shifted = po.run_jobs(model, [po.SeqJob(chunk, np.arange(40), None, pos0=delta)])[0]
        for l in range(spec.n_layers):
            assert rel_err(shifted.k[l], ref.k[l]) < 1e-10
            assert rel_err(shifted.v[l], ref.v[l]) < 1e-10


def test_legolink0_compile_drops_dummies(tiny):
    spec, w, model = tiny
    chunk = pi.gen_tokens(30, spec.vocab, 16)
    (k0, v0), = po.compile_chunks(model, [chunk], n_dummy=4)
    fr = po.full_prefill(model, np.concatenate([np.zeros(4, dtype=np.int32), chunk]))
    for l in range(spec.n_layers):
        assert k0[l].shape[0] == 30
        assert rel_err(k0[l], fr.k[l][4:]) < 1e-12
    # the dummies matter: without them the KV differs
    (k1, _), = po.compile_chunks(model, [chunk], n_dummy=0)
    assert rel_err(k1[1], k0[1]) > 1e-6


# ----------------------------------------------------------------------------- brute-force twin

@pytest.mark.parametrize("k,n_dummy,lens", [(2, 0, [5, 16, 19]), (0, 4, [7, 9]), (17, 0, [18, 3, 20])])
def test_matches_bruteforce(micro, k, n_dummy, lens):
    spec, w, model = micro
    chunks = [pi.gen_tokens(L, spec.vocab, 21, i) for i, L in enumerate(lens)]
    q = pi.gen_tokens(5, spec.vocab, 22)
    _, _, out = _link(spec, model, chunks, [q], k=k, n_dummy=n_dummy)
    bm = bf.BruteModel(spec, w)
    comp = [bf.brute_compile(bm, c, n_dummy) for c in chunks]
    ref = bf.brute_link(bm, comp, chunks, q, k)
    assert list(out.meta[0].selected) == ref["selected"]
    assert rel_err(out.hidden[0], np.array(ref["hidden"])) < 1e-12
    assert rel_err(out.logits[0][0], np.array(ref["logits"])) < 1e-12
    for l in range(spec.n_layers):
        assert rel_err(out.k[0][l], np.array(ref["k"][l])) < 1e-12
        assert rel_err(out.v[0][l], np.array(ref["v"][l])) < 1e-12


# ----------------------------------------------------------------------------- metadata

def test_metadata_hand_example():
    g = json.load(open(os.path.join(GOLD, "tiny_link_metadata.json")))
    st = po.OracleStore(None, 64)
    cids = [st._add_chunk(np.zeros(L, dtype=np.int32), [], []) for L in g["chunk_lengths"]]
    assert [st.chunks[c].blocks for c in cids] == g["compile_blocks"]
    m, = st.plan([(cids, g["query_length"])], g["k"])
    assert m.private_blocks.tolist() == g["private_blocks"]
    assert m.selected.tolist() == g["selected"]
    assert m.slots.tolist() == g["slots"]
    assert m.page_table.tolist() == g["page_table"]
    assert m.page_pos.tolist() == g["page_pos"]
    assert m.page_len.tolist() == g["page_len"]


@pytest.mark.parametrize("k", [0, 1, 2, 15, 16, 17, 32, 512])
def test_metadata_closed_forms(k):
    lens = [512, 37, 16, 1, 100]
    lq = 21
    st = po.OracleStore(None, 1000)
    cids = [st._add_chunk(np.zeros(L, dtype=np.int32), [], []) for L in lens]
    m, = st.plan([(cids, lq)], k)
    ceil = lambda a: -(-a // 16)
    assert len(m.selected) == sum(min(k, L) for L in lens) + lq
    assert len(m.page_table) == sum(ceil(L) for L in lens) + ceil(lq)
    assert len(m.private_blocks) == sum(ceil(min(k, L)) for L in lens) + ceil(lq)
    assert np.all(np.diff(m.selected) > 0)
    assert sum(m.page_len) == sum(lens) + lq
    # every selected row's slot lies in the page that holds its position
    for s, slot in zip(m.selected, m.slots):
        j = int(np.searchsorted(m.page_pos, s, side="right") - 1)
        assert slot // 16 == m.page_table[j] and slot % 16 == s - m.page_pos[j]
        assert slot // 16 in set(m.private_blocks.tolist())
    # shared blocks of the chunks stay in the table past each chunk's private prefix
    off = 0
    for c, L in zip(cids, lens):
        j0 = int(np.searchsorted(m.page_pos, off))
        for j in range(ceil(min(k, L)), ceil(L)):
            assert m.page_table[j0 + j] == st.chunks[c].blocks[j]
        off += L


def test_allocator_all_or_nothing_and_refcounts():
    st = po.OracleStore(None, 10)
    a = st._add_chunk(np.zeros(64, dtype=np.int32), [], [])      # blocks 0-3
    b = st._add_chunk(np.zeros(40, dtype=np.int32), [], [])      # blocks 4-6
    free_before = set(st.free)
    with pytest.raises(po.OutOfBlocks):
        st.plan([([a, b], 16), ([a, b], 16)], 16)                 # needs 6, only 3 free
    assert st.free == free_before
    m, = st.plan([([a, b], 16)], 16)
    assert m.private_blocks.tolist() == [7, 8, 9]
    st.requests[0] = (m.private_blocks.tolist(), [a, b])
    st.chunks[a].refs += 1
    st.chunks[b].refs += 1
    st.release_chunk(a)                                            # still referenced by the request
    assert a in st.chunks and not (set(range(4)) & st.free)
    st.release_request(0)
    assert a not in st.chunks and set(range(4)) <= st.free and {7, 8, 9} <= st.free


# ----------------------------------------------------------------------------- decode after link

def test_decode_after_full_recompute_is_prefill(tiny, micro):
    """k >= every chunk length: each decoded token equals the last row of a plain prefill of
    prompt + query + the tokens decoded so far (hidden state, logits and its K/V)."""
    for spec, w, model in (tiny, micro):
        lens = [64, 40, 64] if spec is pi.TINY else [5, 16, 19]
        chunks = [pi.gen_tokens(L, spec.vocab, 41, i) for i, L in enumerate(lens)]
        q = pi.gen_tokens(16 if spec is pi.TINY else 6, spec.vocab, 42)   # tiny: the first token opens a block
        st, _, out = _link(spec, model, chunks, [q], k=max(lens))
        seq = np.concatenate(chunks + [q])
        for t in pi.gen_tokens(3, spec.vocab, 43):
            d = st.decode(out.rids, [int(t)])
            seq = np.append(seq, t)
            fr = po.full_prefill(model, seq)
            assert d.positions.tolist() == [len(seq) - 1]
            assert rel_err(d.hidden[0], fr.hidden[-1]) < 1e-11
            assert rel_err(d.logits[0], model.logits(fr.hidden[-1:])[0]) < 1e-11
            for l in range(spec.n_layers):
                assert rel_err(d.k[0][l], fr.k[l][-1]) < 1e-11
                assert rel_err(d.v[0][l], fr.v[l][-1]) < 1e-11


def test_decode_single_chunk_k0_is_prefill(tiny):
    """One chunk, k = 0: the linked KV is the chunk's own prefill, so decoding continues a
    plain prefill of chunk + query."""
    spec, w, model = tiny
    chunk, q = pi.gen_tokens(50, spec.vocab, 44), pi.gen_tokens(9, spec.vocab, 45)
    st, _, out = _link(spec, model, [chunk], [q], k=0)
    seq = np.concatenate([chunk, q])
    for t in pi.gen_tokens(2, spec.vocab, 46):
        d = st.decode(out.rids, [int(t)])
        seq = np.append(seq, t)
        fr = po.full_prefill(model, seq)
        assert rel_err(d.hidden[0], fr.hidden[-1]) < 1e-11
        assert rel_err(d.logits[0], model.logits(fr.hidden[-1:])[0]) < 1e-11


@pytest.mark.parametrize("k,n_dummy,lens", [(2, 0, [5, 16, 19]), (0, 4, [7, 9]), (17, 0, [18, 3, 20])])
def test_decode_matches_bruteforce(micro, k, n_dummy, lens):
    """Between the special cases: decoding after LegoLink-k agrees with the per-token twin,
    which generates from the caches its own link left behind."""
    spec, w, model = micro
    chunks = [pi.gen_tokens(L, spec.vocab, 47, i) for i, L in enumerate(lens)]
    q = pi.gen_tokens(5, spec.vocab, 48)
    gen = [int(t) for t in pi.gen_tokens(3, spec.vocab, 49)]
    st, _, out = _link(spec, model, chunks, [q], k=k, n_dummy=n_dummy)
    ds = [st.decode(out.rids, [t]) for t in gen]
    bm = bf.BruteModel(spec, w)
    comp = [bf.brute_compile(bm, c, n_dummy) for c in chunks]
    ref = bf.brute_link(bm, comp, chunks, q, k, decode=gen)
    for i, d in enumerate(ds):
        assert d.positions.tolist() == [sum(lens) + len(q) + i]
        assert rel_err(d.hidden[0], np.array(ref["decode_hidden"][i])) < 1e-12
        assert rel_err(d.logits[0], np.array(ref["decode_logits"][i])) < 1e-12
        for l in range(spec.n_layers):
            assert rel_err(d.k[0][l], np.array(ref["decode_k"][i][l])) < 1e-12
            assert rel_err(d.v[0][l], np.array(ref["decode_v"][i][l])) < 1e-12


def test_decode_metadata_hand_example(tiny):
    spec, w, model = tiny
    g = json.load(open(os.path.join(GOLD, "tiny_decode_metadata.json")))
    st = po.OracleStore(model, 64)
    chunks = [pi.gen_tokens(L, spec.vocab, 50, i) for i, L in enumerate(g["chunk_lengths"])]
    cids = st.compile_many(chunks)
    assert [st.chunks[c].blocks for c in cids] == g["compile_blocks"]
    reqs = [([cids[c] for c in r["chunks"]], pi.gen_tokens(r["query_length"], spec.vocab, 51, i))
            for i, r in enumerate(g["requests"])]
    out = st.link(reqs, 2)
    for m, r in zip(out.meta, g["requests"]):
        assert m.private_blocks.tolist() == r["link_private_blocks"]
        assert m.page_table.tolist() == r["link_page_table"]
        assert m.page_pos.tolist() == r["link_page_pos"]
        assert m.page_len.tolist() == r["link_page_len"]
    order = [out.rids[i] for i in g["decode_order"]]
    for i, step in enumerate(g["decode_steps"]):
        d = st.decode(order, [i + 1] * len(order))
        assert d.positions.tolist() == step["positions"] and d.slots.tolist() == step["slots"]
    for rid, f in zip(out.rids, g["final"]):
        m = st.request_meta(rid)
        for key in ("page_table", "page_pos", "page_len", "private_blocks"):
            assert getattr(m, key).tolist() == f[key], key
    # the link's own returned metadata is not changed by decoding
    assert out.meta[0].page_table.tolist() == g["requests"][0]["link_page_table"]


def test_decode_requests_are_independent(tiny):
    """Decoding several requests in one call gives each the result it gets alone."""
    spec, w, model = tiny
    chunks = [pi.gen_tokens(L, spec.vocab, 52, i) for i, L in enumerate([64, 23, 40])]
    queries = [pi.gen_tokens(Lq, spec.vocab, 53, i) for i, Lq in enumerate([16, 7])]
    st, cids, out = _link(spec, model, chunks, queries, k=3)
    both = st.decode(out.rids[::-1], [5, 6])
    for i, (q, tok) in enumerate(zip(queries, [6, 5])):
        st1, _, o1 = _link(spec, model, chunks, [q], k=3)
        d1 = st1.decode(o1.rids, [tok])
        j = 1 - i
        assert both.positions[j] == d1.positions[0]
        assert rel_err(both.hidden[j], d1.hidden[0]) < 1e-13
        assert rel_err(both.logits[j], d1.logits[0]) < 1e-13


def test_decode_allocation_all_or_nothing(tiny):
    spec, w, model = tiny
    chunk = pi.gen_tokens(32, spec.vocab, 54)
    st, cids, out = _link(spec, model, [chunk], [pi.gen_tokens(16, spec.vocab, 55)] * 2, k=2, num_blocks=6)
    assert len(st.free) == 0                          # 2 chunk blocks + 2 x (1 private + 1 query)
    before = [st.request_meta(r).page_len.tolist() for r in out.rids]
    with pytest.raises(po.OutOfBlocks):
        st.decode(out.rids, [1, 2])                   # both last pages are full
    assert [st.request_meta(r).page_len.tolist() for r in out.rids] == before
    with pytest.raises(ValueError):
        st.decode([out.rids[0]] * 2, [1, 2])
    st.release_request(out.rids[1])
    d = st.decode(out.rids[:1], [3])                  # the released blocks serve the next page
    assert d.slots.tolist() == [min(out.meta[1].private_blocks) * 16]


# ----------------------------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes(monkeypatch, micro):
    """Each plausible slip in the oracle makes at least one pin fail."""
    spec, w, model = micro
    toks = pi.gen_tokens(23, spec.vocab, 31)
    hid_ref = tr.prefill(spec, w, toks)[0].numpy()

    def fails(patch_target, bad):
        with monkeypatch.context() as m:
            m.setattr(po, patch_target, bad)
            got = po.full_prefill(po.OracleModel(spec, w), toks)
        return rel_err(got.hidden, hid_ref) > 1e-6

    good_rope, good_att = po.rope, po.causal_attention

    def rope_wrong_sign(x, pos, base):
        return good_rope(x, -pos, base)

    def rope_interleaved(x, pos, base):
        y = x.reshape(*x.shape[:-1], -1, 2).swapaxes(-1, -2).reshape(x.shape)
        return good_rope(y, pos, base)

    def att_strict_mask(q, k, v, qp, kp):
        out = good_att(q, k, v, qp, kp + 0.5)  # a row no longer sees itself
        out[0] = 0.0
        return out

    def att_wrong_group(q, k, v, qp, kp):
        G = k.shape[1]
        return good_att(q, k[:, ::-1].copy(), v[:, ::-1].copy(), qp, kp) if G > 1 else good_att(q, k, v, qp, kp)

    assert fails("rope", rope_wrong_sign)
    assert fails("rope", rope_interleaved)
    assert fails("causal_attention", att_strict_mask)
    assert fails("causal_attention", att_wrong_group)
    with monkeypatch.context() as m:
        m.setattr(po, "silu", lambda x: x)
        assert rel_err(po.full_prefill(po.OracleModel(spec, w), toks).hidden, hid_ref) > 1e-6


def test_decode_pins_catch_planted_mistakes(monkeypatch, tiny):
    """Slips in the oracle's decode bookkeeping make the decode pins fail: reading the
    compiled KV where the link recomputed rows, an off-by-one position, and forgetting the
    rows decoded earlier."""
    spec, w, model = tiny
    lens = [64, 40, 64]
    chunks = [pi.gen_tokens(L, spec.vocab, 41, i) for i, L in enumerate(lens)]
    q = pi.gen_tokens(16, spec.vocab, 42)
    gen = [int(t) for t in pi.gen_tokens(3, spec.vocab, 43)]

    def worst_error():
        st, _, out = _link(spec, model, chunks, [q], k=max(lens))
        seq, worst = np.concatenate(chunks + [q]), 0.0
        for t in gen:
            d = st.decode(out.rids, [t])
            seq = np.append(seq, t)
            worst = max(worst, rel_err(d.hidden[0], po.full_prefill(model, seq).hidden[-1]))
        return worst

    assert worst_error() < 1e-11
    good_kv = po.OracleStore._request_kv

    def compiled_rows_only(self, rid, l):
        K, V = good_kv(self, rid, l)
        st, off = self.linked[rid], 0
        for c in st.chunk_ids:             # undo the link's recomputed rows
            ch = self.chunks[c]
            K[off:off + len(ch.tokens)] = po._f64(ch.k[l])
            V[off:off + len(ch.tokens)] = po._f64(ch.v[l])
            off += len(ch.tokens)
        return K, V

    def no_decoded_rows(self, rid, l):
        K, V = good_kv(self, rid, l)
        n_dec = len(self.linked[rid].k_dec[l])
        if n_dec:
            K[-n_dec:] = 0.0
            V[-n_dec:] = 0.0
        return K, V

    for bad in (compiled_rows_only, no_decoded_rows):
        with monkeypatch.context() as m:
            m.setattr(po.OracleStore, "_request_kv", bad)
            assert worst_error() > 1e-6, bad.__name__
    good_jobs = po.run_jobs

    def reuses_last_position(model_, jobs):
        """The new token takes the request's last used position instead of the next one."""
        out = []
        for j in jobs:
            if len(j.sel) == 1 and j.base_kv is not None:
                n = int(j.sel[0])
                toks = np.concatenate([j.tokens[:n - 1], j.tokens[n:n + 1]])
                out.append(po.SeqJob(toks, np.array([n - 1]), lambda l, f=j.base_kv: tuple(a[:-1] for a in f(l))))
            else:
                out.append(j)
        return good_jobs(model_, out)

    with monkeypatch.context() as m:
        m.setattr(po, "run_jobs", reuses_last_position)
        assert worst_error() > 1e-6


def test_decode_opens_blocks_in_call_order(tiny):
    """Two requests whose last pages are full decode in one call: the new blocks are taken in
    the call's request order (hand-worked fixture)."""
    spec, w, model = tiny
    g = json.load(open(os.path.join(GOLD, "tiny_decode_two_new_blocks.json")))
    st = po.OracleStore(model, 64)
    cids = st.compile_many([pi.gen_tokens(L, spec.vocab, 56, i) for i, L in enumerate(g["chunk_lengths"])])
    assert [st.chunks[c].blocks for c in cids] == g["compile_blocks"]
    out = st.link([([cids[c] for c in r["chunks"]], pi.gen_tokens(r["query_length"], spec.vocab, 57, i))
                   for i, r in enumerate(g["requests"])], 2)
    assert [m.private_blocks.tolist() for m in out.meta] == [r["link_private_blocks"] for r in g["requests"]]
    for i, step in enumerate(g["steps"]):
        d = st.decode([out.rids[j] for j in step["order"]], [i + 3] * len(step["order"]))
        assert d.positions.tolist() == step["positions"] and d.slots.tolist() == step["slots"]
    for rid, f in zip(out.rids, g["final"]):
        m = st.request_meta(rid)
        assert {k: getattr(m, k).tolist() for k in f} == f


# ----------------------------------------------------------------------------- dynamic selection (CacheBlend-r)

def test_dynamic_scores_match_bruteforce(micro):
    """Layer-0 attention mass per prompt token: the vectorised oracle equals the per-token loop."""
    spec, w, model = micro
    lens = [5, 16, 19]
    chunks = [pi.gen_tokens(L, spec.vocab, 31, i) for i, L in enumerate(lens)]
    q = pi.gen_tokens(6, spec.vocab, 32)
    bm = bf.BruteModel(spec, w)
    comp = [bf.brute_compile(bm, c) for c in chunks]
    got = po.query_attention_scores(model, chunks, [np.asarray(ck[0]) for ck, _ in comp], q)
    ref = np.asarray(bf.brute_scores(bm, comp, chunks, q))
    assert got.shape == (sum(lens),)
    assert rel_err(got, ref) < 1e-12
    # every query row's weights sum to one over the prompt and the query keys it sees
    assert 0.0 < got.sum() < len(q) * spec.n_heads


def test_dynamic_select_hand_example():
    """Top r % of N by score, equal scores taking the lower position first, ascending output."""
    sc = np.array([1.0, 3.0, 3.0, 2.0, 0.0])
    assert po.select_top(sc, 0).tolist() == []
    assert po.select_top(sc, 20).tolist() == [1]          # n = 1: of the tied 3.0s, position 1
    assert po.select_top(sc, 40).tolist() == [1, 2]
    assert po.select_top(sc, 60).tolist() == [1, 2, 3]
    assert po.select_top(sc, 99).tolist() == [0, 1, 2, 3]  # n = floor(4.95) = 4
    assert po.select_top(sc, 100).tolist() == [0, 1, 2, 3, 4]


def test_dynamic_metadata_hand_example():
    """Blocks of recomputed tokens inside a chunk become private copies (hand-worked ids)."""
    g = json.load(open(os.path.join(GOLD, "tiny_dynamic_metadata.json")))
    st = po.OracleStore(None, 64)
    cids = [st._add_chunk(np.zeros(g["chunk_len"], dtype=np.int32), [], []) for _ in range(g["n_chunks"])]
    m, = st.plan_selected([(cids, g["query_len"], g["chosen"])])
    for key in ("private_blocks", "page_table", "page_pos", "page_len", "selected", "slots"):
        assert getattr(m, key).tolist() == g[key], key


def test_selected_first_k_equals_legolink_k(tiny):
    """Choosing the first k tokens of every chunk reproduces LegoLink-k exactly (metadata and outputs)."""
    spec, w, model = tiny
    lens = [64, 37, 64, 5]
    chunks = [pi.gen_tokens(L, spec.vocab, 33, i) for i, L in enumerate(lens)]
    q = pi.gen_tokens(16, spec.vocab, 34)
    for k in (2, 17):
        st_a, cids_a, out_a = _link(spec, model, chunks, [q], k=k)
        st_b = po.OracleStore(model, 256)
        cids_b = st_b.compile_many(chunks)
        out_b = st_b.link_selected([(cids_b, q, [list(range(min(k, L))) for L in lens])])
        for key in ("selected", "slots", "page_table", "page_pos", "page_len", "private_blocks"):
            assert np.array_equal(getattr(out_a.meta[0], key), getattr(out_b.meta[0], key)), key
        assert rel_err(out_b.hidden[0], out_a.hidden[0]) < 1e-13
        assert rel_err(out_b.logits[0], out_a.logits[0]) < 1e-13


def test_selected_matches_bruteforce(micro):
    """Recomputed rows chosen anywhere in a chunk: equal to the per-token loop recomputing them."""
    spec, w, model = micro
    lens = [5, 16, 19]
    chosen = [[3], [0, 7, 15], [2, 18]]
    chunks = [pi.gen_tokens(L, spec.vocab, 35, i) for i, L in enumerate(lens)]
    q = pi.gen_tokens(5, spec.vocab, 36)
    st = po.OracleStore(model, 256)
    cids = st.compile_many(chunks)
    out = st.link_selected([(cids, q, chosen)])
    bm = bf.BruteModel(spec, w)
    comp = [bf.brute_compile(bm, c) for c in chunks]
    ref = bf.brute_link(bm, comp, chunks, q, 0, chosen=chosen)
    assert list(out.meta[0].selected) == ref["selected"]
    assert rel_err(out.hidden[0], np.array(ref["hidden"])) < 1e-12
    assert rel_err(out.logits[0][0], np.array(ref["logits"])) < 1e-12
    for l in range(spec.n_layers):
        assert rel_err(out.k[0][l], np.array(ref["k"][l])) < 1e-12


def test_dynamic_r100_is_full_recompute(tiny):
    """r = 100 %: every prompt token is recomputed -- a plain prefill of the concatenated prompt."""
    spec, w, model = tiny
    chunks = [pi.gen_tokens(64, spec.vocab, 37, i) for i in range(3)]
    q = pi.gen_tokens(16, spec.vocab, 38)
    st = po.OracleStore(model, 256)
    cids = st.compile_many(chunks)
    out, scores = st.link_dynamic([(cids, q)], 100, all_logits=True)
    assert out.meta[0].selected.tolist() == list(range(3 * 64 + 16))
    fr = po.full_prefill(model, np.concatenate(chunks + [q]))
    assert rel_err(out.hidden[0], fr.hidden[-16:]) < 1e-11
    for l in range(spec.n_layers):
        assert rel_err(out.k[0][l], fr.k[l]) < 1e-11


def test_dynamic_r0_is_naive_reuse(micro):
    """r = 0: nothing but the query is recomputed -- every chunk's compiled KV reused as it is
    (the per-token loop with k = 0 and no dummy prefix)."""
    spec, w, model = micro
    lens = [5, 16, 19]
    chunks = [pi.gen_tokens(L, spec.vocab, 39, i) for i, L in enumerate(lens)]
    q = pi.gen_tokens(5, spec.vocab, 40)
    st = po.OracleStore(model, 256)
    cids = st.compile_many(chunks)
    out, _ = st.link_dynamic([(cids, q)], 0)
    bm = bf.BruteModel(spec, w)
    comp = [bf.brute_compile(bm, c) for c in chunks]
    ref = bf.brute_link(bm, comp, chunks, q, 0)
    assert out.meta[0].selected.tolist() == ref["selected"] == list(range(40, 45))
    assert rel_err(out.hidden[0], np.array(ref["hidden"])) < 1e-12


def test_dynamic_selects_by_attention(micro):
    """The chosen rows are the highest-scoring ones: each chosen token's score is at least every
    unchosen one's (ties to the lower position), and their count is floor(r N / 100)."""
    spec, w, model = micro
    lens = [5, 16, 19]
    chunks = [pi.gen_tokens(L, spec.vocab, 41, i) for i, L in enumerate(lens)]
    q = pi.gen_tokens(5, spec.vocab, 42)
    st = po.OracleStore(model, 256)
    cids = st.compile_many(chunks)
    out, (sc,) = st.link_dynamic([(cids, q)], 15)
    N = sum(lens)
    chosen = [u for u in out.meta[0].selected.tolist() if u < N]
    assert len(chosen) == 15 * N // 100
    rest = [u for u in range(N) if u not in chosen]
    assert min(sc[chosen]) >= max(sc[rest])
