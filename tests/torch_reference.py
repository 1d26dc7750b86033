"""Independent library-routine formulation of the decoder, used only to pin the oracle.

It computes a plain causal prefill with torch's own building blocks in float64:
scaled_dot_product_attention (is_causal) for attention, rms_norm for the norms,
silu/linear for the MLP, and RoPE written as complex multiplication
(x_i + j*x_{i+D/2}) * exp(j*p*theta_i) rather than the oracle's sin/cos form.
It shares no code with the oracle or the CUDA library.
"""
import torch
import torch.nn.functional as F


def complex_rope(x: torch.Tensor, pos: torch.Tensor, base: float) -> torch.Tensor:
    """x [n, heads, D] (float64) rotated by complex multiplication at positions pos [n]."""
    D = x.shape[-1]
    theta = 1.0 / (base ** (torch.arange(0, D, 2, dtype=torch.float64) / D))
    rot = torch.polar(torch.ones(len(pos), D // 2, dtype=torch.float64),
                      pos.to(torch.float64)[:, None] * theta[None, :])
    z = torch.complex(x[..., : D // 2], x[..., D // 2:]) * rot[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def prefill(spec, weights, tokens):
    """Final-normed hidden [N, d], last-row logits and per-layer pre-RoPE K, V of a causal prefill."""
    f = lambda t: t.detach().to(torch.float64)
    H, G, D = spec.n_heads, spec.n_kv_heads, spec.head_dim
    tok = torch.as_tensor(tokens, dtype=torch.long)
    N = len(tok)
    pos = torch.arange(N)
    h = f(weights["embed"])[tok]
    ks, vs = [], []
    for l in range(spec.n_layers):
        W = {n: f(weights[f"layers.{l}.{n}"]) for n in
             ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")}
        x = F.rms_norm(h, (spec.d_model,), W["attn_norm"], spec.rms_eps)
        q = F.linear(x, W["wq"]).view(N, H, D)
        k = F.linear(x, W["wk"]).view(N, G, D)
        v = F.linear(x, W["wv"]).view(N, G, D)
        ks.append(k)
        vs.append(v)
        qr = complex_rope(q, pos, spec.rope_base).transpose(0, 1)                  # [H, N, D]
        kr = complex_rope(k, pos, spec.rope_base).repeat_interleave(H // G, dim=1).transpose(0, 1)
        vr = v.repeat_interleave(H // G, dim=1).transpose(0, 1)
        o = F.scaled_dot_product_attention(qr, kr, vr, is_causal=True)           # [H, N, D]
        h = h + F.linear(o.transpose(0, 1).reshape(N, H * D), W["wo"])
        x = F.rms_norm(h, (spec.d_model,), W["mlp_norm"], spec.rms_eps)
        h = h + F.linear(F.silu(F.linear(x, W["w_gate"])) * F.linear(x, W["w_up"]), W["w_down"])
    hid = F.rms_norm(h, (spec.d_model,), f(weights["final_norm"]), spec.rms_eps)
    logits = F.linear(hid[-1:], f(weights["lm_head"]))
    return hid, logits, ks, vs
