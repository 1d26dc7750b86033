"""GPU parity of the CUDA path against the fp64 CPU oracle, through the C ABI.

Element-by-element comparisons on seeded inputs: the tcgen05 and SIMT GEMMs, the
fused-RoPE paged attention, and whole compile + link runs (tiny fp32 config at 1e-4,
small bf16 GQA models at 2e-2), including ragged chunks, several requests, repeated
chunks, k = 0 with the LegoLink-0 dummy prefix, k larger than a chunk, decode steps after
the link (page growth across block boundaries), and the error paths of the store.
"""
import numpy as np
import pytest
import torch

import pic_inputs as pi
from oracle import pic_oracle as po
from tests.helpers import compare_link, library_run, oracle_run, rel_err, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    from position_independent_kv_link_gb300 import load
    load()


# ----------------------------------------------------------------------------- GEMM

@pytest.mark.parametrize("N,K,T", [(128, 64, 1), (256, 128, 5), (128, 4096, 224), (6144, 4096, 224),
                                   (384, 512, 300), (256, 1024, 513), (4096, 14336, 64), (1024, 256, 16)])
def test_gemm_bf16_tcgen05(N, K, T):
    from position_independent_kv_link_gb300 import gemm
    W = pi.randn((N, K), ("gemmW", N, K), 0.05, torch.bfloat16)
    X = pi.randn((T, K), ("gemmX", T, K), 1.0, torch.bfloat16)
    Y = gemm(W.cuda(), X.cuda())
    torch.cuda.synchronize()
    ref = X.double() @ W.double().T
    assert rel_err(Y, ref) < 1e-5


@pytest.mark.parametrize("N,K,T", [(128, 64, 1), (6144, 4096, 224), (384, 512, 300), (4096, 14336, 64),
                                   (1024, 256, 513), (256, 2048, 137), (512, 64, 129), (512, 256, 1100),
                                   (256, 1024, 1024), (384, 128, 1500), (1024, 4096, 1100)])
def test_gemm_bf16_packed_weights(N, K, T):
    """The layout the model repacks its matrices into, through the packed tcgen05 path: (1024,
    256, 513) over three token tiles, (256, 2048, 137) two weight tiles split over 64 CTAs,
    (512, 64, 129) one k-block per tile; from 1024 token rows with 256-row weight tiles when N
    allows: (512, 256, 1100) over five token tiles (the last ragged), (256, 1024, 1024) one
    weight tile, (1024, 4096, 1100) ~8 k-blocks per CTA over 64-k-block tiles (ranges that end
    with a shorter segment are walked from it); (384, 128, 1500) stays at 128 rows (N not a
    multiple of 256)."""
    from position_independent_kv_link_gb300 import gemm_packed, pack_weight
    W = pi.randn((N, K), ("gemmWp", N, K), 0.05, torch.bfloat16)
    X = pi.randn((T, K), ("gemmXp", T, K), 1.0, torch.float16)
    Y = gemm_packed(pack_weight(W.cuda()), N, K, X.cuda())
    torch.cuda.synchronize()
    assert rel_err(Y, X.double() @ W.double().T) < 1e-5


@pytest.mark.parametrize("N,K,T", [(96, 64, 7), (768, 256, 24), (1024, 512, 300)])
def test_gemm_f32_simt(N, K, T):
    from position_independent_kv_link_gb300 import gemm
    W = pi.randn((N, K), ("gemmWf", N, K), 0.05)
    X = pi.randn((T, K), ("gemmXf", T, K), 1.0)
    Y = gemm(W.cuda(), X.cuda())
    torch.cuda.synchronize()
    assert rel_err(Y, X.double() @ W.double().T) < 1e-5


# ----------------------------------------------------------------------------- attention

def _attn_case(dtype, D, H, G, lens, qlen, k_first, seed):
    """Pages of ragged chunks + a query, random pre-RoPE K/V, queries at selected rows."""
    rng = np.random.default_rng(seed)
    pblk, ppos, plen = [], [], []
    off = 0
    sel = []
    for i, L in enumerate(lens + [qlen]):
        for j in range(-(-L // 16)):
            pblk.append(len(pblk))
            ppos.append(off + 16 * j)
            plen.append(min(16, L - 16 * j))
        sel += list(range(off, off + (min(k_first, L) if i < len(lens) else L)))
        off += L
    sel = sorted(set(sel))
    nb = len(pblk)
    perm = rng.permutation(nb + 3)[:nb]               # scattered physical blocks
    pblk = [int(perm[i]) for i in range(nb)]
    K = pi.randn((nb + 3, G, 16, D), ("attK", seed), 1.0, dtype)
    V = pi.randn((nb + 3, G, 16, D), ("attV", seed), 1.0, dtype)
    q = pi.randn((len(sel), H, D), ("attQ", seed), 1.0, torch.float32)
    return q, np.array(sel), K, V, (np.array(pblk), np.array(ppos), np.array(plen)), off


@pytest.mark.parametrize("dtype,D,H,G", [(torch.float32, 64, 4, 4), (torch.float32, 128, 8, 2),
                                         (torch.bfloat16, 128, 8, 2), (torch.bfloat16, 128, 32, 8),
                                         (torch.bfloat16, 64, 4, 1), (torch.bfloat16, 128, 8, 8),
                                         (torch.bfloat16, 128, 8, 4), (torch.bfloat16, 128, 16, 2)])
def test_paged_attention_fused_rope(dtype, D, H, G):
    from position_independent_kv_link_gb300 import attention, rope_table
    base = 500000.0 if D == 128 else 10000.0
    q, qpos, K, V, pages, n_pos = _attn_case(dtype, D, H, G, [37, 16, 5, 100, 64], 20, 3, 7)
    rope = rope_table(n_pos + 8, D, base)
    out = attention(q.cuda(), qpos, K.cuda(), V.cuda(), pages, rope, G)
    torch.cuda.synchronize()
    # oracle: assemble K/V in position order, rotate at absolute positions, causal softmax
    blk, ppos, plen = pages
    Ka = np.concatenate([K[b, :, :n].double().numpy().transpose(1, 0, 2) for b, n in zip(blk, plen)])
    Va = np.concatenate([V[b, :, :n].double().numpy().transpose(1, 0, 2) for b, n in zip(blk, plen)])
    pos = np.concatenate([np.arange(p, p + n) for p, n in zip(ppos, plen)])
    ref = po.causal_attention(po.rope(q.double().numpy(), qpos, base), po.rope(Ka, pos, base), Va, qpos, pos)
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    assert rel_err(out, ref) < tol


def test_paged_attention_config2_shape():
    """The 8B link's attention at its full size: 10 x 512 chunks + 64 query, k = 16
    (224 query rows, 324 pages, 32 Q / 8 KV heads), split over page runs as in the link."""
    from position_independent_kv_link_gb300 import attention, rope_table
    q, qpos, K, V, pages, n_pos = _attn_case(torch.bfloat16, 128, 32, 8, [512] * 10, 64, 16, 11)
    rope = rope_table(n_pos + 16, 128, 500000.0)
    out = attention(q.cuda(), qpos, K.cuda(), V.cuda(), pages, rope, 8)
    torch.cuda.synchronize()
    blk, ppos, plen = pages
    Ka = np.concatenate([K[b, :, :n].double().numpy().transpose(1, 0, 2) for b, n in zip(blk, plen)])
    Va = np.concatenate([V[b, :, :n].double().numpy().transpose(1, 0, 2) for b, n in zip(blk, plen)])
    pos = np.concatenate([np.arange(p, p + n) for p, n in zip(ppos, plen)])
    ref = po.causal_attention(po.rope(q.double().numpy(), qpos, 500000.0), po.rope(Ka, pos, 500000.0), Va, qpos, pos)
    assert rel_err(out, ref) < 2e-2


# ----------------------------------------------------------------------------- whole link

@pytest.fixture(scope="module")
def tiny():
    spec = pi.TINY
    w = pi.gen_weights(spec, gains="random")
    from position_independent_kv_link_gb300 import PicModel
    return spec, w, PicModel(spec, w), po.OracleModel(spec, w)


def _store(model, nb=256, rows=2048, reqs=16, pos=8192, lg=64):
    from position_independent_kv_link_gb300 import PicStore
    return PicStore(model, num_blocks=nb, max_rows=rows, max_requests=reqs, max_positions=pos, max_logit_rows=lg)


def test_tiny_config_link(tiny):
    spec, w, model, om = tiny
    wl = pi.config_workloads()["tiny"]
    store = _store(model)
    _, res = library_run(store, wl)
    _, _, out = oracle_run(om, wl, 256)
    compare_link(store, res, out, spec)


@pytest.mark.parametrize("k,n_dummy", [(0, 0), (0, 4), (1, 0), (2, 0), (16, 0), (17, 0), (1000, 0)])
def test_tiny_link_variants(tiny, k, n_dummy):
    """Ragged chunks (not multiples of 16), 3 requests with repeats, several k."""
    spec, w, model, om = tiny
    wl = pi.make_workload("ragged", spec, 5, [37, 64, 5, 16, 50], 19, k, n_requests=3, n_dummy=n_dummy)
    wl.requests[1].chunk_ids = [4, 0, 0, 2]
    wl.requests[2].chunk_ids = [3]
    wl.requests[2].query = wl.requests[2].query[:1]
    store = _store(model)
    _, res = library_run(store, wl, all_logits=True)
    _, _, out = oracle_run(om, wl, 256, all_logits=True)
    compare_link(store, res, out, spec)


@pytest.fixture(scope="module")
def small_bf16():
    spec = pi.SMALL_BF16
    w = pi.gen_weights(spec, gains="random")
    from position_independent_kv_link_gb300 import PicModel
    return spec, w, PicModel(spec, w), po.OracleModel(spec, w)


@pytest.mark.parametrize("k,n_dummy", [(16, 0), (2, 0), (0, 4), (40, 0)])
def test_small_bf16_link(small_bf16, k, n_dummy):
    spec, w, model, om = small_bf16
    wl = pi.make_workload("small", spec, 6, [128, 77, 200, 16, 33, 128], 40, k, n_requests=2, n_dummy=n_dummy)
    wl.requests[1].chunk_ids = [5, 1, 3, 0]
    store = _store(model)
    _, res = library_run(store, wl)
    _, _, out = oracle_run(om, wl, 256)
    compare_link(store, res, out, spec)


def test_small_bf16_link_batch_of_four(small_bf16):
    """Four requests in one tensor-core batch (ragged queries, shared and repeated chunks, the
    same chunk at different offsets): every request's hidden states, logits and recomputed K/V
    rows of every layer are compared, so a row offset or work-item boundary that only goes wrong
    for a later request of the batch shows."""
    spec, w, model, om = small_bf16
    wl = pi.make_workload("small batch", spec, 8, [128, 77, 200, 16, 33, 128, 300, 64], 40, 16, n_requests=4)
    wl.requests[1].chunk_ids = [5, 1, 3, 0]
    wl.requests[2].chunk_ids = [7, 6, 2]
    wl.requests[2].query = wl.requests[2].query[:23]
    wl.requests[3].chunk_ids = [4, 0, 6, 1, 5, 3, 2, 7]
    wl.requests[3].query = wl.requests[3].query[:1]
    store = _store(model, lg=128)
    _, res = library_run(store, wl, all_logits=True)
    _, _, out = oracle_run(om, wl, 256, all_logits=True)
    errs = compare_link(store, res, out, spec)
    assert all(f"k{i}.1" in errs for i in range(4))


# ----------------------------------------------------------------------------- decode after link

def _decode_parity(store, om, wl, steps, seed, nb=256):
    """Links the workload in the library and in the oracle, then runs `steps` decode steps over
    every request (in reverse request order). Each step: positions, slots and page tables
    bit-exact; hidden, logits and the new K/V rows of every layer within tolerance."""
    spec = wl.spec
    _, res = library_run(store, wl)
    ost, _, out = oracle_run(om, wl, nb)
    compare_link(store, res, out, spec, check_kv=False)
    lib_r, orc_r = res.requests[::-1], out.rids[::-1]
    worst_all = 0.0
    for step in range(steps):
        toks = [int(t) for t in pi.gen_tokens(len(lib_r), spec.vocab, seed, step)]
        d = store.decode(lib_r, toks)
        store.sync()
        o = ost.decode(orc_r, toks)
        assert np.array_equal(d.positions, o.positions) and np.array_equal(d.slots, o.slots), step
        for lr, orid in zip(lib_r, orc_r):
            info, m = store.request_info(lr), ost.request_meta(orid)
            for key in ("page_table", "page_pos", "page_len", "private_blocks"):
                assert np.array_equal(info[key], getattr(m, key)), (step, key, info[key], getattr(m, key))
        errs = {"hidden": rel_err(d.hidden, o.hidden), "logits": rel_err(d.logits, o.logits)}
        for l in range(spec.n_layers):
            k, v = store.kv_rows(l, d.slots)
            errs[f"k{l}"] = rel_err(k, np.stack([kk[l] for kk in o.k]))
            errs[f"v{l}"] = rel_err(v, np.stack([vv[l] for vv in o.v]))
        worst = max(errs, key=errs.get)
        assert errs[worst] <= tol_for(spec), (step, worst, errs[worst])
        worst_all = max(worst_all, errs[worst])
    return worst_all


def test_tiny_decode_after_link(tiny):
    """3 requests over ragged chunks with 16, 19 and 16 query rows: steps 1 and 17 open a new
    block for two requests at once (the call order decides the ids), step 14 for one."""
    spec, w, model, om = tiny
    wl = pi.make_workload("ragged decode", spec, 5, [37, 64, 5, 16, 50], 16, 2, n_requests=3)
    wl.requests[1].chunk_ids = [4, 0, 0, 2]
    wl.requests[1].query = pi.gen_tokens(19, spec.vocab, 60)
    wl.requests[2].chunk_ids = [3]
    _decode_parity(_store(model), om, wl, 18, 61)


@pytest.mark.parametrize("k,n_dummy", [(16, 0), (0, 4)])
def test_small_bf16_decode_after_link(small_bf16, k, n_dummy):
    """bf16 GQA (4 query heads per KV head, D = 128: the tensor-core attention) with 2 decode
    rows per step, far fewer than one 32-row work item."""
    spec, w, model, om = small_bf16
    wl = pi.make_workload("small decode", spec, 6, [128, 77, 200, 16, 33, 128], 40, k, n_requests=2,
                          n_dummy=n_dummy)
    wl.requests[1].chunk_ids = [5, 1, 3, 0]
    _decode_parity(_store(model), om, wl, 10, 62)


def test_decode_errors_leave_state_unchanged(tiny):
    from position_independent_kv_link_gb300 import PicError
    from position_independent_kv_link_gb300 import _lib as L
    spec, w, model, om = tiny
    store = _store(model, nb=6)
    a, = store.compile([np.arange(32) % spec.vocab])                 # 2 blocks
    q = np.arange(16, dtype=np.int32)
    res = store.link([([a], q), ([a], q)], 2)                        # 2 x (1 private + 1 query): pool full
    r0, r1 = res.requests
    info = [store.request_info(r) for r in (r0, r1)]
    for bad, status in ((([r0, r1], [1, 2]), L.PIC_ERR_OUT_OF_BLOCKS), ((([r0, r0], [1, 2])), L.PIC_ERR_INVALID_ARG),
                        ((([r0, 999], [1, 2])), L.PIC_ERR_INVALID_ARG), ((([r0], [spec.vocab])), L.PIC_ERR_INVALID_ARG)):
        with pytest.raises(PicError) as e:
            store.decode(*bad)
        assert e.value.status == status
        assert store.free_blocks() == 0
        for r, before in zip((r0, r1), info):
            after = store.request_info(r)
            assert all(np.array_equal(after[k], before[k]) for k in before)
    store.release_request(r1)
    d = store.decode([r0], [5])                                      # takes the lowest freed block
    store.sync()
    assert d.slots.tolist() == [int(min(info[1]["private_blocks"])) * 16]
    assert d.positions.tolist() == [48]


# ----------------------------------------------------------------------------- store error paths

def test_store_errors_leave_state_unchanged(tiny):
    from position_independent_kv_link_gb300 import PicError
    from position_independent_kv_link_gb300 import _lib as L
    spec, w, model, om = tiny
    store = _store(model, nb=10)
    a, b = store.compile([np.arange(64) % spec.vocab, np.arange(40) % spec.vocab])   # 4 + 3 blocks
    assert store.free_blocks() == 3
    with pytest.raises(PicError) as e:
        store.link([([a, b], np.zeros(16, dtype=np.int32))] * 2, 16)
    assert e.value.status == L.PIC_ERR_OUT_OF_BLOCKS and store.free_blocks() == 3
    with pytest.raises(PicError) as e:
        store.compile([np.array([spec.vocab])])
    assert e.value.status == L.PIC_ERR_INVALID_ARG and store.free_blocks() == 3
    with pytest.raises(PicError) as e:
        store.link([([a, 999], np.zeros(4, dtype=np.int32))], 2)
    assert e.value.status == L.PIC_ERR_INVALID_ARG
    res = store.link([([a, b], np.zeros(16, dtype=np.int32))], 16)
    assert store.free_blocks() == 0
    store.release_chunk(a)                    # still used by the request
    assert store.free_blocks() == 0
    store.release_request(res.requests[0])    # frees 3 private blocks and chunk a's 4
    assert store.free_blocks() == 7
    store.release_chunk(b)
    assert store.free_blocks() == 10
    store.sync()
