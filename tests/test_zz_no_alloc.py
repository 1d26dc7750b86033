"""The allocation-free attention call matches the regular one.

pic_op_attention_noalloc serves callers that cannot allocate device memory (code
inside a memory pool it does not own, hosts that forbid cudaMalloc after start-up,
paths that must not synchronize the device): it keeps its scratch in a fixed area of
the library instead of a caller buffer. This file is collected last on purpose, and it
must pass both on its own in a fresh process and after every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import pic_inputs as pi
from oracle import pic_oracle as po
from tests.helpers import rel_err

pytestmark = pytest.mark.gpu


def _case(seed):
    """Ragged chunks + a query over scattered pages (bf16 KV, 8 Q / 2 KV heads, head_dim 128; fp32 q)."""
    rng = np.random.default_rng(seed)
    lens, qlen = [300, 37, 512, 16, 200], 40
    pblk, ppos, plen, sel = [], [], [], []
    off = 0
    for i, L in enumerate(lens + [qlen]):
        for j in range(-(-L // 16)):
            pblk.append(len(pblk))
            ppos.append(off + 16 * j)
            plen.append(min(16, L - 16 * j))
        sel += list(range(off, off + (min(3, L) if i < len(lens) else L)))
        off += L
    nb = len(pblk) + 5
    pblk = [int(b) for b in rng.permutation(nb)[:len(pblk)]]
    K = pi.randn((nb, 2, 16, 128), ("noallocK", seed), 1.0, torch.bfloat16).cuda()
    V = pi.randn((nb, 2, 16, 128), ("noallocV", seed), 1.0, torch.bfloat16).cuda()
    q = pi.randn((len(sel), 8, 128), ("noallocQ", seed), 1.0, torch.float32).cuda()
    i32 = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return q, i32(sel), K, V, i32(pblk), i32(ppos), i32(plen), off


def _oracle(q, qpos, K, V, blk, ppos, plen, base):
    """fp64 oracle attention of the case: K/V gathered in position order, RoPE at absolute positions."""
    Ka = np.concatenate([K[b, :, :n].double().cpu().numpy().transpose(1, 0, 2) for b, n in zip(blk, plen)])
    Va = np.concatenate([V[b, :, :n].double().cpu().numpy().transpose(1, 0, 2) for b, n in zip(blk, plen)])
    pos = np.concatenate([np.arange(p, p + n) for p, n in zip(ppos, plen)])
    return po.causal_attention(po.rope(q.double().cpu().numpy(), qpos, base), po.rope(Ka, pos, base), Va, qpos, pos)


def test_noalloc_attention_matches_regular_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    from position_independent_kv_link_gb300 import _lib as L, api
    lib = L.load()
    assert lib.pic_op_attention_noalloc_max_scratch() == 16 << 20
    stream = torch.cuda.current_stream()
    sp = C.c_void_p(stream.cuda_stream)
    P = lambda a: a.ctypes.data_as(L.PI32)
    for seed in (1, 2):                          # two calls in a row on the shared area
        q, qpos, K, V, blk, ppos, plen, n_pos = _case(seed)
        T, n_pages = q.shape[0], len(blk)
        # the case's pages are split into runs whose partial results are merged, so the
        # partial-result regions of the fixed area are in use
        counts = np.zeros(3, dtype=np.int32)
        items = np.zeros((4096, 7), dtype=np.int32)
        combs = np.zeros((4096, 5), dtype=np.int32)
        seq_rows, seq_pages = np.array([0, T], dtype=np.int32), np.array([0, n_pages], dtype=np.int32)
        L.check(lib.pic_op_attention_plan(L.PIC_BF16, 8, 2, 128, 1, P(seq_rows), P(seq_pages), P(qpos), P(ppos),
                                          torch.cuda.get_device_properties(0).multi_processor_count,
                                          P(items), 4096, P(combs), 4096, P(counts)))
        assert counts[1] > 0
        rope = api.rope_table(n_pos + 16, 128, 500000.0)
        ref = torch.empty(q.shape, dtype=torch.float16, device="cuda")
        nb = lib.pic_op_attention_scratch_bytes(T, 8, 2, 128, n_pages)
        scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
        L.check(lib.pic_op_attention(L.PIC_BF16, T, 8, 2, 128, q.data_ptr(), P(qpos), K.data_ptr(), V.data_ptr(),
                                     P(blk), P(ppos), P(plen), n_pages, K.shape[0], rope.data_ptr(), rope.shape[0],
                                     ref.data_ptr(), scratch.data_ptr(), nb, sp))
        assert lib.pic_sync(None, sp) == L.PIC_OK
        got = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
        L.check(lib.pic_op_attention_noalloc(L.PIC_BF16, T, 8, 2, 128, q.data_ptr(), P(qpos), K.data_ptr(),
                                             V.data_ptr(), P(blk), P(ppos), P(plen), n_pages, K.shape[0],
                                             rope.data_ptr(), rope.shape[0], got.data_ptr(), sp))
        # a bounded wait given up inside the kernels would surface here, at the call that caused it
        assert lib.pic_sync(None, sp) == L.PIC_OK
        # same plan, same kernels, same inputs: the outputs are identical bit for bit
        assert torch.equal(got, ref)
        assert rel_err(got, _oracle(q, qpos, K, V, blk, ppos, plen, 500000.0)) < 2e-2


def test_noalloc_attention_rejects_oversized_work():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    from position_independent_kv_link_gb300 import _lib as L, api
    lib = L.load()
    # T rows whose rotated fp16 q (the tensor-core path's operand: T x 32 heads x 128 dims x 2
    # bytes) alone fills the fixed area; the metadata and merge partials come on top of it,
    # whatever the work plan
    T = int(lib.pic_op_attention_noalloc_max_scratch()) // (32 * 128 * 2)
    n_pages = T // 16
    qpos = np.arange(T, dtype=np.int32)
    blk = np.arange(n_pages, dtype=np.int32)
    ppos = (16 * np.arange(n_pages)).astype(np.int32)
    plen = np.full(n_pages, 16, dtype=np.int32)
    q = torch.zeros((T, 32, 128), dtype=torch.float32, device="cuda")
    K = torch.zeros((n_pages, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    rope = api.rope_table(16 * n_pages + 16, 128, 500000.0)
    out = torch.zeros((T, 32, 128), dtype=torch.float16, device="cuda")
    P = lambda a: a.ctypes.data_as(L.PI32)
    st = lib.pic_op_attention_noalloc(L.PIC_BF16, T, 32, 8, 128, q.data_ptr(), P(qpos), K.data_ptr(), K.data_ptr(),
                                      P(blk), P(ppos), P(plen), n_pages, n_pages, rope.data_ptr(), rope.shape[0],
                                      out.data_ptr(), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == L.PIC_ERR_CAPACITY
    assert b"fixed area" in lib.pic_last_error()
