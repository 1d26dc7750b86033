"""Host logic of the paged attention: the work plan (pic_op_attention_plan, no GPU needed).

The plan cuts every (row block, KV head) of a batch into page runs. Whatever the cut, the
attention is only right if every page a block can see is read exactly once and every split
run's partial result is merged exactly once; these invariants are checked on link, decode and
compile-shaped batches, ragged and random, for each kernel family's shape. The part-size rule
of the persistent kernel (a few candidate sizes, the one whose snake deal over the CTAs has
the smallest estimated makespan plus merge cost) is restated here independently and compared
item by item.
"""

import numpy as np
import pytest
import torch

BLOCK = 16


@pytest.fixture(scope="module")
def lib():
    from position_independent_kv_link_gb300 import _lib as L
    return L.load()


def _plan(*a, **k):
    from position_independent_kv_link_gb300 import attention_plan
    return attention_plan(*a, **k)


# ----------------------------------------------------------------------------- batch layouts

def link_seq(lens, qlen, k):
    """Rows and pages of one linked request: first min(k, L) rows of each chunk + the query."""
    rows, pages, off = [], [], 0
    for i, L in enumerate(list(lens) + [qlen]):
        pages += [off + BLOCK * j for j in range(-(-L // BLOCK))]
        rows += list(range(off, off + (min(k, L) if i < len(lens) else L)))
        off += L
    return rows, pages


def decode_seq(lens, qlen):
    """One decode row after a link: the row at the next position, its page appended if new."""
    n = sum(lens) + qlen
    _, pages = link_seq(lens, qlen, 0)
    if qlen % BLOCK == 0:
        pages = pages + [n]
    return [n], pages


def compile_seqs(lens):
    return [(list(range(L)), [BLOCK * j for j in range(-(-L // BLOCK))]) for L in lens]


def random_batch(rng, n_seq, kind):
    seqs = []
    for _ in range(n_seq):
        lens = [int(x) for x in rng.integers(1, 600, size=int(rng.integers(1, 6)))]
        qlen = int(rng.integers(1, 70))
        if kind == "decode":
            seqs.append(decode_seq(lens, qlen))
        else:
            seqs.append(link_seq(lens, qlen, int(rng.choice([0, 1, 2, 16, 17, 32, 1000]))))
    return seqs


SHAPES = {   # name: (dtype, H, G, D) -> the kernel family that runs it
    "tcgen05": (torch.bfloat16, 32, 8, 128),
    "mma_rep1": (torch.bfloat16, 8, 8, 128),
    "mma_rep8": (torch.bfloat16, 16, 2, 128),
    "simt": (torch.float32, 4, 4, 64),
}
ROWS_PER_BLOCK = {"tcgen05": 64, "mma_rep1": 32, "mma_rep8": 16, "simt": 16}


# ----------------------------------------------------------------------------- invariants

def expected_blocks(seqs, rb):
    """(row0, nrows, page_begin, page_end, page_end of the first 32 rows) per row block,
    indices over the concatenated batch."""
    out, r_off, p_off = [], 0, 0
    for rows, pages in seqs:
        for b0 in range(0, len(rows), rb):
            n = min(rb, len(rows) - b0)
            pe = sum(1 for p in pages if p <= rows[b0 + n - 1])
            pe0 = sum(1 for p in pages if p <= rows[b0 + min(n, 32) - 1])
            out.append((r_off + b0, n, p_off, p_off + pe, p_off + pe0))
        r_off += len(rows)
        p_off += len(pages)
    return out


def check_plan(items, combs, n_parts, seqs, G, rb, num_sms, persistent):
    blocks = expected_blocks(seqs, rb)
    pe0_of = {(row0, nrows): pe0 for row0, nrows, _, _, pe0 in blocks}
    by_key = {}
    for it in items.tolist():
        row0, nrows, g, p0, p1, part, pmid = it
        assert 0 <= g < G and 1 <= nrows <= rb and p0 <= p1
        # the first 32 rows see the run's pages up to page_mid, none after it
        assert pmid == min(p1, max(p0, pe0_of[(row0, nrows)]))
        by_key.setdefault((row0, nrows, g), []).append((p0, p1, part))
    assert len(by_key) == len(blocks) * G, "every (row block, KV head) has items, and nothing else does"
    comb_by_key = {}
    for c in combs.tolist():
        row0, nrows, g, part0, nparts = c
        assert (row0, nrows, g) not in comb_by_key
        comb_by_key[(row0, nrows, g)] = (part0, nparts)
    seen_parts = []
    for row0, nrows, pb, pe, _ in blocks:
        for g in range(G):
            runs = sorted(by_key[(row0, nrows, g)])
            # the runs tile [pb, pe) exactly: each page read once
            assert runs[0][0] == pb and runs[-1][1] == pe
            assert all(a[1] == b[0] for a, b in zip(runs, runs[1:]))
            if len(runs) == 1:
                assert runs[0][2] == -1 and (row0, nrows, g) not in comb_by_key
                continue
            part0, nparts = comb_by_key[(row0, nrows, g)]
            assert nparts == len(runs)
            assert sorted(r[2] for r in runs) == list(range(part0, part0 + nparts))
            # runs are cut from the block's start in equal sizes (whole tiles when persistent)
            sizes = [r[1] - r[0] for r in runs]
            assert len(set(sizes[:-1])) <= 1 and sizes[-1] <= sizes[0]
            if persistent:
                assert sizes[0] % 4 == 0
            seen_parts += [r[2] for r in runs]
    assert sorted(seen_parts) == list(range(n_parts)), "every partial result merged exactly once"
    assert len(comb_by_key) == len(combs)
    # scratch bounds the library sizes its buffers by
    assert n_parts <= 4 * num_sms + G * len(blocks)
    assert len(items) <= n_parts + G * len(blocks)


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("num_sms", [1, 7, 152])
def test_plan_invariants_on_method_batches(lib, shape, num_sms):
    dtype, H, G, D = SHAPES[shape]
    batches = {
        "8B link 10x512 + 64, k=16": [link_seq([512] * 10, 64, 16)],
        "8B link k=32": [link_seq([512] * 10, 64, 32)],
        "full recompute": [link_seq([512] * 4, 64, 512)],
        "LegoLink-0": [link_seq([512] * 10, 64, 0)],
        "decode after link": [decode_seq([512] * 10, 64)],
        "decode, 5 requests": [decode_seq([300, 37, 16], 5), decode_seq([512] * 3, 16), decode_seq([1], 1),
                               decode_seq([999], 47), decode_seq([64, 64], 64)],
        "compile batch": compile_seqs([512, 512, 37, 1]),
        "link, ragged, 3 requests": [link_seq([37, 64, 5, 16, 50], 19, 2), link_seq([50, 37, 37, 5], 19, 2),
                                     link_seq([16], 3, 2)],
    }
    for name, seqs in batches.items():
        items, combs, n_parts = _plan(dtype, H, G, D, seqs, num_sms)
        check_plan(items, combs, n_parts, seqs, G, ROWS_PER_BLOCK[shape], num_sms, shape == "tcgen05")


@pytest.mark.parametrize("kind", ["link", "decode"])
@pytest.mark.parametrize("seed", range(6))
def test_plan_invariants_random_batches(lib, kind, seed):
    rng = np.random.default_rng(seed)
    seqs = random_batch(rng, int(rng.integers(1, 6)), kind)
    for shape, (dtype, H, G, D) in SHAPES.items():
        num_sms = int(rng.choice([1, 5, 152]))
        items, combs, n_parts = _plan(dtype, H, G, D, seqs, num_sms)
        check_plan(items, combs, n_parts, seqs, G, ROWS_PER_BLOCK[shape], num_sms, shape == "tcgen05")


# ----------------------------------------------------------------------------- the part-size rule

def model_plan(seqs, G, rb, num_sms, persistent):
    """Independent restatement of the planner's rule (same item fields and order)."""
    blocks = expected_blocks(seqs, rb)
    total = sum(pe - pb for _, _, pb, pe, _ in blocks)

    def build(P):
        items, parts = [], 0
        for row0, n, pb, pe, pe0 in blocks:
            ns = max(1, -(-(pe - pb) // P))
            for g in range(G):
                if ns == 1:
                    items.append((row0, n, g, pb, pe, -1, pe0))
                    continue
                for s in range(ns):
                    p0, p1 = pb + s * P, min(pe, pb + (s + 1) * P)
                    items.append((row0, n, g, p0, p1, parts + s, min(p1, max(p0, pe0))))
                parts += ns
        return sorted(items, key=lambda it: -(it[4] - it[3])), parts   # stable: heaviest first

    def cost(it):
        """In 0.01 us: 26 per 64-key tile, 33 per MMA tile taking part in it (rows 0-31 up to
        page_mid, rows 32-63 throughout), 491 per item."""
        nt = (it[4] - it[3] + 3) // 4
        n0 = max(0, (it[6] - it[3] + 3) // 4)
        n1 = nt if it[1] > 32 else 0
        return 26 * nt + 33 * (n0 + n1) + 491

    if not persistent:
        target = max(1, (4 * num_sms) // G)
        return build(max(4, -(-total // target)))[0]

    def snake(items):
        n = min(len(items), num_sms)
        dealt, load = [None] * len(items), [0] * max(1, n)
        for k0 in range(0, len(items), n):
            m = min(n, len(items) - k0)
            for c in range(m):
                it = items[k0 + (m - 1 - c if (k0 // n) & 1 else c)]
                dealt[k0 + c] = it
                load[c] += cost(it)
        return dealt, max(load)

    max_pages = max([pe - pb for _, _, pb, pe, _ in blocks] + [1])

    def n_items(P):
        return G * sum(max(1, -(-(pe - pb) // P)) for _, _, pb, pe, _ in blocks)

    cands = set()
    for per_sm in (1, 1.5, 2, 3, 4):
        want = max(1, int(per_sm * 2) * num_sms // 2)
        P = (max(8, -(-total * G // want)) + 3) // 4 * 4   # from the average page count
        cands.add(P)
        while n_items(P) > want and P < max_pages:           # the smallest size that fits the target
            P += 4
        cands.add(P)
    best = None
    for P in sorted(cands):
        items, parts = build(P)
        dealt, span = snake(items)
        est = span * num_sms + 150 * parts   # makespan + the merge (150 per split part, over the SMs)
        if best is None or (est, len(dealt)) < (best[0], len(best[1])):
            best = (est, dealt)
    return best[1]


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("num_sms", [3, 152])
def test_plan_follows_the_rule(lib, shape, num_sms):
    dtype, H, G, D = SHAPES[shape]
    rng = np.random.default_rng(11)
    for seqs in ([link_seq([512] * 10, 64, 16)], [decode_seq([512] * 10, 64)], [link_seq([512] * 30, 64, 16)],
                 random_batch(rng, 4, "link"), random_batch(rng, 3, "decode"), compile_seqs([512, 100])):
        items, _, _ = _plan(dtype, H, G, D, seqs, num_sms)
        ref = model_plan(seqs, G, ROWS_PER_BLOCK[shape], num_sms, shape == "tcgen05")
        assert [tuple(it) for it in items.tolist()] == ref


def test_plan_decode_one_item_per_sm(lib):
    """The 8B decode step (one row over 325 pages, 8 KV heads, 152 SMs): 2600 page-units cut
    into 20-page runs (17 per head) give 136 items, at most one per SM."""
    items, combs, n_parts = _plan(torch.bfloat16, 32, 8, 128, [decode_seq([512] * 10, 64)], 152)
    assert len(items) == 136 and n_parts == 136 and len(combs) == 8
    assert max(it[4] - it[3] for it in items.tolist()) == 20


# ----------------------------------------------------------------------------- argument checks

def test_plan_rejects_bad_input_and_reports_sizes(lib):
    from position_independent_kv_link_gb300 import _lib as L
    rows, pages = link_seq([512] * 10, 64, 16)
    arr = lambda a: np.ascontiguousarray(a, dtype=np.int32)
    seq_rows, seq_pages, rp, pp = arr([0, len(rows)]), arr([0, len(pages)]), arr(rows), arr(pages)
    counts = np.zeros(3, dtype=np.int32)
    P = lambda a: a.ctypes.data_as(L.PI32)

    def call(sr, sp, r, p, num_sms=152):
        return lib.pic_op_attention_plan(L.PIC_BF16, 32, 8, 128, 1, P(sr), P(sp), P(r), P(p), num_sms,
                                         None, 0, None, 0, P(counts))
    # output arrays too small: the sizes are reported for a second call (the c2 link: 4 blocks x 8
    # KV heads in 56-page parts, 152 items for 152 SMs, all of them split)
    assert call(seq_rows, seq_pages, rp, pp) == L.PIC_ERR_CAPACITY and counts.tolist() == [152, 32, 152]
    bad = rp.copy()
    bad[5] = bad[4]                                            # row positions must ascend
    assert call(seq_rows, seq_pages, bad, pp) == L.PIC_ERR_INVALID_ARG
    assert call(arr([1, len(rows)]), seq_pages, rp, pp) == L.PIC_ERR_INVALID_ARG   # offsets start at 0
    assert call(seq_rows, seq_pages, rp, pp, num_sms=0) == L.PIC_ERR_INVALID_ARG
