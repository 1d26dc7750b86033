"""Shared test helpers: error metric and oracle/library runs on the same seeded inputs."""
import numpy as np
import torch

import pic_inputs as pi
from oracle import pic_oracle as po


def rel_err(got, ref) -> float:
    """max |got - ref| / max |ref| (the tolerance metric of the parity tests)."""
    g = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    r = ref.detach().double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    return float(np.max(np.abs(g - r)) / max(1e-300, float(np.max(np.abs(r)))))


def tol_for(spec) -> float:
    return 1e-4 if spec.dtype == "f32" else 2e-2


def library_run(store, wl, all_logits=False, compile_kwargs=None):
    """Compile every chunk of the workload then link all its requests in one batch."""
    cids = store.compile(wl.chunks, n_dummy=wl.n_dummy, **(compile_kwargs or {}))
    reqs = [([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests]
    res = store.link(reqs, wl.k, all_logits=all_logits)
    store.sync()
    return cids, res


def oracle_run(model, wl, num_blocks, all_logits=False):
    st = po.OracleStore(model, num_blocks)
    cids = st.compile_many(wl.chunks, wl.n_dummy)
    out = st.link([([cids[c] for c in r.chunk_ids], r.query) for r in wl.requests], wl.k, all_logits=all_logits)
    return st, cids, out


def compare_link(store, res, out, spec, check_kv=True, layers=None):
    """Metadata bit-exact; hidden, logits and every recomputed K/V row within tolerance."""
    tol = tol_for(spec)
    errs = {}
    n0 = 0
    for i, r in enumerate(res.requests):
        info = store.request_info(r)
        m = out.meta[i]
        for key in ("selected", "slots", "page_table", "page_pos", "page_len", "private_blocks"):
            assert np.array_equal(info[key], getattr(m, key)), (i, key, info[key][:20], getattr(m, key)[:20])
        lq = out.hidden[i].shape[0]
        errs[f"hidden{i}"] = rel_err(res.hidden[n0:n0 + lq], out.hidden[i])
        n0 += lq
        if check_kv:
            for l in (range(spec.n_layers) if layers is None else layers):
                k, v = store.kv_rows(l, info["slots"])
                errs[f"k{i}.{l}"] = rel_err(k, out.k[i][l])
                errs[f"v{i}.{l}"] = rel_err(v, out.v[i][l])
    lg_ref = np.concatenate(out.logits, 0)
    errs["logits"] = rel_err(res.logits, lg_ref)
    worst = max(errs, key=errs.get)
    assert errs[worst] <= tol, (worst, errs[worst], tol)
    return errs
