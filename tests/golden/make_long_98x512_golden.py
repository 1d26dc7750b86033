"""Writes the fp64 oracle's outputs of the long-context link (8B shape, 98 x 512-token
chunks + 64-token query, k = 16, all 32 layers) to tests/golden/long_98x512_link_outputs.npz.

Calls only the oracle (oracle/pic_oracle.py) and the seeded input generators (pic_inputs):
the weights are the seeded random-init 8B weights, the compiled chunk KV is the seeded
stand-in that the GPU test imports into the library (pic_inputs.gen_chunk_kv, one seed per
chunk). Stored: the final-normed hidden states of the 64 query rows, the logits of the last
query row, and the recomputed K/V of a sample of selected rows at a sample of layers, all as
float32 (the comparison tolerance is 2e-2 relative, far above float32 rounding).

Takes ~15-30 minutes and ~35 GB of host memory:  python tests/golden/make_long_98x512_golden.py
"""
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import pic_inputs as pi  # noqa: E402
from oracle import pic_oracle as po  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "long_98x512_link_outputs.npz")
# recomputed rows and layers whose K/V are stored (rows index the selected list, ascending positions)
KV_ROWS = [0, 15, 16, 800, 1551, 1552, 1567, 1568, 1600, 1631]
KV_LAYERS = [0, 1, 15, 31]


def main():
    t0 = time.time()
    spec = pi.LLAMA3_8B
    wl = pi.config_workloads()["8b_98x512"]
    w = pi.gen_weights(spec)
    om = po.OracleModel(spec, w)
    ost = po.OracleStore(om, 1 << 13)
    ids = {}
    for c in range(len(wl.chunks)):
        k, v = pi.gen_chunk_kv(spec, len(wl.chunks[c]), c)
        ids[c] = ost.import_chunk(wl.chunks[c], [k[l] for l in range(spec.n_layers)],
                                  [v[l] for l in range(spec.n_layers)])
    print(f"inputs ready in {time.time() - t0:.0f} s", flush=True)
    r = wl.requests[0]
    out = ost.link([([ids[c] for c in r.chunk_ids], r.query)], wl.k)
    print(f"link done in {time.time() - t0:.0f} s", flush=True)
    np.savez(OUT,
             hidden=out.hidden[0].astype(np.float32),
             logits=out.logits[0].astype(np.float32),
             selected=out.meta[0].selected,
             kv_rows=np.asarray(KV_ROWS, dtype=np.int32),
             kv_layers=np.asarray(KV_LAYERS, dtype=np.int32),
             k=np.stack([out.k[0][l][KV_ROWS] for l in KV_LAYERS]).astype(np.float32),
             v=np.stack([out.v[0][l][KV_ROWS] for l in KV_LAYERS]).astype(np.float32))
    print(f"wrote {OUT}", flush=True)


if __name__ == "__main__":
    main()
