"""An independent fp64 torch-CPU statement of the decoder layer, used to pin the oracle.

It follows the module structure of page "12 · 从 Transformer 到 LLaMA 系列" §八 (norm ->
attention -> residual, norm -> SwiGLU -> residual; KV heads repeated along dim 1 before
the attention), with the even/odd rotation of page "第 10 章：现代 LLaMA 架构" §3 in place
of that page's half-split one, and torch's own ``scaled_dot_product_attention`` with
``is_causal=True`` as the library routine for the attention.  Written for this test suite;
shares no code with the oracle.
"""
import torch
import torch.nn.functional as F


def _norm(x, g, eps):
    return g * (x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + eps))


def _rotate_pairs(x, cos, sin):
    ev, od = x[..., 0::2], x[..., 1::2]
    return torch.stack((ev * cos - od * sin, ev * sin + od * cos), dim=-1).flatten(-2)


def block(x, w, cos, sin, n_heads, n_kv_heads, eps):
    """x: [B, S, d] fp64 tensor at positions 0..S-1; w: dict of fp64 tensors [out, in]."""
    B, S, d = x.shape
    D = w["wq"].shape[0] // n_heads
    xn = _norm(x, w["attn_norm"], eps)
    q = F.linear(xn, w["wq"]).view(B, S, n_heads, D).transpose(1, 2)
    k = F.linear(xn, w["wk"]).view(B, S, n_kv_heads, D).transpose(1, 2)
    v = F.linear(xn, w["wv"]).view(B, S, n_kv_heads, D).transpose(1, 2)
    c, s = cos[:S], sin[:S]
    q, k = _rotate_pairs(q, c, s), _rotate_pairs(k, c, s)
    rep = n_heads // n_kv_heads
    o = F.scaled_dot_product_attention(q, k.repeat_interleave(rep, dim=1),
                                       v.repeat_interleave(rep, dim=1), is_causal=True)
    h = x + F.linear(o.transpose(1, 2).reshape(B, S, n_heads * D), w["wo"])
    hn = _norm(h, w["ffn_norm"], eps)
    return h + F.linear(F.silu(F.linear(hn, w["w_gate"])) * F.linear(hn, w["w_up"]), w["w_down"])


def model(tokens, layers, final_norm, embed, lm_head, cos, sin, n_heads, n_kv_heads, eps):
    x = F.embedding(tokens, embed)
    for w in layers:
        x = block(x, w, cos, sin, n_heads, n_kv_heads, eps)
    return F.linear(_norm(x, final_norm, eps), lm_head)
