"""Brute-force twin of the oracle: compile and LegoLink link as explicit per-token loops.

TEST INFRASTRUCTURE ONLY (imported by tests alone). It shares no code with
`pic_oracle` and uses no matrix routine: every dot product, norm and softmax is a
Python loop over plain floats, and tokens are processed one at a time in position
order, each attending to the per-layer KV cache of the positions before it. Only for
tiny shapes.

Method (cited by page title and section):
  compile: prefill each chunk alone from position 0, keep per-layer pre-RoPE K and V
           ("EPIC: Efficient Position-Independent Caching ...", atlas.scime.ai summary,
           Approach; dummy prefix of LegoLink-0 from its Measured effects table).
  link:    the first k tokens of every chunk and the query are recomputed through every
           layer, every other row reuses its compiled KV; RoPE is applied to each key
           at attention time from its absolute position ("MEPIC: Memory Efficient
           Position Independent Caching for LLM Serving", abstract).
  decode:  after the link, each further token takes the next position and runs through
           every layer against the linked caches, which it extends.
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple


def _rows(t) -> List[List[float]]:
    import torch
    return t.detach().to(torch.float64).tolist()


class BruteModel:
    def __init__(self, spec, weights):
        self.spec = spec
        self.E = _rows(weights["embed"])
        self.Wlm = _rows(weights["lm_head"])
        self.gf = _rows(weights["final_norm"])
        self.L = []
        for l in range(spec.n_layers):
            p = f"layers.{l}."
            self.L.append({n: _rows(weights[p + n]) for n in
                           ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")})


def _norm(x, g, eps):
    ms = 0.0
    for a in x:
        ms += a * a
    r = 1.0 / math.sqrt(ms / len(x) + eps)
    return [x[i] * r * g[i] for i in range(len(x))]


def _mv(W, x):
    out = []
    for row in W:
        acc = 0.0
        for i in range(len(x)):
            acc += row[i] * x[i]
        out.append(acc)
    return out


def _turn(vec, p, base):
    """Rotate one head vector: dim i pairs with dim i + D/2, angle p * base^(-2i/D)."""
    D = len(vec)
    h = D // 2
    out = [0.0] * D
    for i in range(h):
        a = p * base ** (-2.0 * i / D)
        c, s = math.cos(a), math.sin(a)
        out[i] = vec[i] * c - vec[i + h] * s
        out[i + h] = vec[i + h] * c + vec[i] * s
    return out


def _step(m: BruteModel, tok: int, p: int, Kc, Vc) -> List[float]:
    """Run one token at position p through all layers; writes its K/V into the caches.

    Kc[l][u] / Vc[l][u]: list over KV heads of pre-RoPE head vectors for position u.
    Returns the final-normed hidden state.
    """
    sp = m.spec
    H, G, D = sp.n_heads, sp.n_kv_heads, sp.head_dim
    rep = H // G
    h = list(m.E[tok])
    for l, W in enumerate(m.L):
        x = _norm(h, W["attn_norm"], sp.rms_eps)
        q, k, v = _mv(W["wq"], x), _mv(W["wk"], x), _mv(W["wv"], x)
        Kc[l][p] = [k[g * D:(g + 1) * D] for g in range(G)]
        Vc[l][p] = [v[g * D:(g + 1) * D] for g in range(G)]
        att = []
        for hq in range(H):
            g = hq // rep
            qr = _turn(q[hq * D:(hq + 1) * D], p, sp.rope_base)
            scores = []
            for u in range(p + 1):
                kr = _turn(Kc[l][u][g], u, sp.rope_base)
                s = 0.0
                for i in range(D):
                    s += qr[i] * kr[i]
                scores.append(s / math.sqrt(D))
            mx = max(scores)
            w = [math.exp(s - mx) for s in scores]
            tot = sum(w)
            o = [0.0] * D
            for u in range(p + 1):
                vu = Vc[l][u][g]
                for i in range(D):
                    o[i] += w[u] / tot * vu[i]
            att += o
        proj = _mv(W["wo"], att)
        h = [h[i] + proj[i] for i in range(len(h))]
        x = _norm(h, W["mlp_norm"], sp.rms_eps)
        a, b = _mv(W["w_gate"], x), _mv(W["w_up"], x)
        act = [a[i] / (1.0 + math.exp(-a[i])) * b[i] for i in range(len(a))]
        dn = _mv(W["w_down"], act)
        h = [h[i] + dn[i] for i in range(len(h))]
    return _norm(h, m.gf, sp.rms_eps)


def brute_compile(m: BruteModel, chunk: Sequence[int], n_dummy: int = 0, dummy: int = 0):
    """Per-token prefill of [dummy * n_dummy, chunk]; returns per layer K, V rows of the chunk."""
    seq = [dummy] * n_dummy + [int(t) for t in chunk]
    nl = m.spec.n_layers
    Kc = [[None] * len(seq) for _ in range(nl)]
    Vc = [[None] * len(seq) for _ in range(nl)]
    for p, tok in enumerate(seq):
        _step(m, tok, p, Kc, Vc)
    return [Kc[l][n_dummy:] for l in range(nl)], [Vc[l][n_dummy:] for l in range(nl)]


def brute_scores(m: BruteModel, compiled: List[Tuple], chunks: Sequence[Sequence[int]],
                 query: Sequence[int]) -> List[float]:
    """Dynamic (attention-based) selection scores, one query token and one head at a time:
    the prompt keeps its compiled layer-0 K; each query token at layer 0 attends causally
    over the prompt and the query tokens up to itself, RoPE at absolute positions; a prompt
    token scores the sum of its softmax weights over the query tokens and heads (the
    reading of CacheBlend's attention-based selection; EPIC summary page)."""
    sp = m.spec
    H, G, D = sp.n_heads, sp.n_kv_heads, sp.head_dim
    rep = H // G
    W = m.L[0]
    K0: List[List[List[float]]] = []          # per position: per KV head pre-RoPE vector
    for (ck, _), c in zip(compiled, chunks):
        K0 += [list(r) for r in ck[0]]
    N = len(K0)
    Q = []
    for tok in query:
        x = _norm(list(m.E[int(tok)]), W["attn_norm"], sp.rms_eps)
        q, k = _mv(W["wq"], x), _mv(W["wk"], x)
        Q.append([q[h * D:(h + 1) * D] for h in range(H)])
        K0.append([k[g * D:(g + 1) * D] for g in range(G)])
    score = [0.0] * N
    for j in range(len(query)):
        p = N + j
        for hq in range(H):
            qr = _turn(Q[j][hq], p, sp.rope_base)
            s = []
            for u in range(p + 1):
                kr = _turn(K0[u][hq // rep], u, sp.rope_base)
                acc = 0.0
                for i in range(D):
                    acc += qr[i] * kr[i]
                s.append(acc / math.sqrt(D))
            mx = max(s)
            w = [math.exp(a - mx) for a in s]
            tot = sum(w)
            for u in range(N):
                score[u] += w[u] / tot
    return score


def brute_link(m: BruteModel, compiled: List[Tuple], chunks: Sequence[Sequence[int]], query: Sequence[int],
               k: int, decode: Sequence[int] = (), chosen: Sequence[Sequence[int]] = None) -> Dict[str, object]:
    """LegoLink-k for one request, one token at a time in position order.

    compiled[i] = (K rows per layer, V rows per layer) of chunk i as brute_compile returns.
    Returns hidden of the query rows, last-row logits and per-layer recomputed K/V rows;
    then the tokens of `decode` are generated one after another from the linked caches
    (their hidden states, logits and per-layer K/V rows under "decode_*"). With `chosen`
    (per chunk the token indices to recompute) those rows are recomputed instead of the
    first k of each chunk.
    """
    nl = m.spec.n_layers
    seq: List[int] = []
    Kc = [[] for _ in range(nl)]
    Vc = [[] for _ in range(nl)]
    selected: List[int] = []
    for i, ((ck, cv), c) in enumerate(zip(compiled, chunks)):
        off = len(seq)
        for t in (range(min(k, len(c))) if chosen is None else sorted(chosen[i])):
            selected.append(off + t)
        seq += [int(t) for t in c]
        for l in range(nl):
            Kc[l] += [list(r) for r in ck[l]]
            Vc[l] += [list(r) for r in cv[l]]
    qoff = len(seq)
    seq += [int(t) for t in query]
    for l in range(nl):
        Kc[l] += [None] * len(query)
        Vc[l] += [None] * len(query)
    selected += list(range(qoff, len(seq)))
    hidden = {}
    for p in selected:
        hidden[p] = _step(m, seq[p], p, Kc, Vc)
    hq = [hidden[p] for p in range(qoff, len(seq))]
    logits = _mv(m.Wlm, hq[-1])
    rk = [[Kc[l][p] for p in selected] for l in range(nl)]
    rv = [[Vc[l][p] for p in selected] for l in range(nl)]
    dh, dl, dk, dv = [], [], [], []
    for tok in decode:
        p = len(seq)
        seq.append(int(tok))
        for l in range(nl):
            Kc[l].append(None)
            Vc[l].append(None)
        dh.append(_step(m, seq[p], p, Kc, Vc))
        dl.append(_mv(m.Wlm, dh[-1]))
        dk.append([Kc[l][p] for l in range(nl)])
        dv.append([Vc[l][p] for l in range(nl)])
    return {"selected": selected, "hidden": hq, "logits": logits, "k": rk, "v": rv,
            "decode_hidden": dh, "decode_logits": dl, "decode_k": dk, "decode_v": dv}
