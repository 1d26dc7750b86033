"""Status plumbing of the device-side checks, with no kernel made to wait or fault.

pic_sync reports what the kernels flagged since the previous pic_sync and clears it:
PIC_ERR_DEVICE_TIMEOUT when a tensor-core kernel gave up a bounded wait, PIC_ERR_RANGE when
a value bound for an fp16 tensor-core operand of a bf16 model left fp16's finite range.
The timeout flags are raised from the host (pic_debug_raise_device_flag), exactly where a
kernel would raise them; the range flag is also raised for real, by inputs whose values are
outside fp16's range (a huge RMSNorm gain, an imported K row, a projection weight).
"""
import numpy as np
import pytest
import torch

import pic_inputs as pi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.set_device(0)
    from position_independent_kv_link_gb300 import _lib as L
    return L, L.load()


def _sync(L, lib):
    import ctypes as C
    return lib.pic_sync(None, C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("which,status", [(1, "PIC_ERR_DEVICE_TIMEOUT"), (2, "PIC_ERR_DEVICE_TIMEOUT"),
                                          (3, "PIC_ERR_RANGE")])
def test_device_flag_reported_once_then_cleared(lib, which, status):
    L, lib_ = lib
    assert _sync(L, lib_) == L.PIC_OK
    assert lib_.pic_debug_raise_device_flag(which) == L.PIC_OK
    assert _sync(L, lib_) == getattr(L, status)
    assert lib_.pic_last_error()           # a message says which check fired
    assert _sync(L, lib_) == L.PIC_OK      # the flag was cleared by the report


def test_device_flag_rejects_unknown(lib):
    L, lib_ = lib
    assert lib_.pic_debug_raise_device_flag(0) == L.PIC_ERR_INVALID_ARG
    assert lib_.pic_debug_raise_device_flag(4) == L.PIC_ERR_INVALID_ARG


def _small_link(spec, w, wl, store_kw=None, chunk_kv=None):
    """Compile (or import) the workload's chunks and link its first request."""
    from position_independent_kv_link_gb300 import PicModel, PicStore
    model = PicModel(spec, w)
    store = PicStore(model, num_blocks=256, max_rows=1024, max_requests=8, max_positions=4096)
    if chunk_kv is None:
        cids = store.compile(wl.chunks)
    else:
        cids = [store.import_chunk(c, *chunk_kv(i, len(c))) for i, c in enumerate(wl.chunks)]
    r = wl.requests[0]
    store.link([([cids[c] for c in r.chunk_ids], r.query)], wl.k)
    return model, store


def test_range_guard_on_a_normed_activation(lib):
    """An RMSNorm gain of 1e5 makes the normed rows (the QKV GEMM's fp16 operand) exceed 65504."""
    L, lib_ = lib
    spec = pi.SMALL_BF16
    wl = pi.make_workload("range", spec, 2, [64, 40], 16, 16)
    w = pi.gen_weights(spec)
    w["layers.0.attn_norm"] = torch.full_like(w["layers.0.attn_norm"], 1e5)
    model, store = _small_link(spec, w, wl)
    with pytest.raises(L.PicError) as e:
        store.sync()
    assert e.value.status == L.PIC_ERR_RANGE
    store.sync()   # reported once
    store.close()
    model.close()
    # the same link with ordinary gains reports nothing
    model, store = _small_link(spec, pi.gen_weights(spec), wl)
    store.sync()
    store.close()
    model.close()


def test_range_guard_on_imported_k(lib):
    """Stored K above 46000 could leave fp16's range once RoPE mixes it with its partner dim."""
    L, lib_ = lib
    spec = pi.SMALL_BF16
    wl = pi.make_workload("range kv", spec, 2, [64, 40], 16, 16)

    def kv(i, n):
        k, v = pi.gen_chunk_kv(spec, n, i)
        if i == 1:
            k[1, 5, 0, 3] = 5e4
        return k.cuda(), v.cuda()
    model, store = _small_link(spec, pi.gen_weights(spec), wl, chunk_kv=kv)
    with pytest.raises(L.PicError) as e:
        store.sync()
    assert e.value.status == L.PIC_ERR_RANGE
    store.close()
    model.close()


def test_range_guard_on_a_weight(lib):
    """A projection weight outside fp16's range cannot be packed: model creation fails."""
    L, lib_ = lib
    from position_independent_kv_link_gb300 import PicModel
    spec = pi.SMALL_BF16
    w = pi.gen_weights(spec)
    w["layers.1.w_up"] = w["layers.1.w_up"].clone()
    w["layers.1.w_up"][3, 7] = 7e4
    with pytest.raises(L.PicError) as e:
        PicModel(spec, w)
    assert e.value.status == L.PIC_ERR_RANGE
    assert _sync(L, lib_) == L.PIC_OK
    assert np.isfinite(w["layers.1.w_up"].float().numpy()).all()
