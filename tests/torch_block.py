"""An independent fp64 torch-CPU statement of the decoder layer, used to pin the oracle.

Written from the layer's equations, not from any page's listing:

    h   = x + Wo · concat_h softmax_causal(q_h k_g(h)ᵀ / √D) v_g(h),  g(h) = h // (H/G)
    out = h + W_down (SiLU(W_gate hn) ⊙ (W_up hn)),  hn = RMSNorm(h)

("05 LLaMA3 Block — 从零件到发动机" §3.1 for the two residual halves; "深度学习进阶（三十）…"
§1.1 for the scaled dot product; "第 10 章：现代 LLaMA 架构" §3 for the even/odd rotation and
§6 for the query heads that share one KV head).  The query heads are indexed as (group,
member) pairs, so each group's keys and values serve its members through an einsum over the
group index: nothing is repeated.  The causal softmax is materialised with torch's own
``softmax``.  Written for this test suite; shares no code with the oracle.
"""
import math

import torch


def _rms(x, g, eps):
    return g * x / torch.sqrt(torch.mean(x * x, dim=-1, keepdim=True) + eps)


def _rotate(x, cos, sin):
    """Even/odd pairs (x[2i], x[2i+1]) of the last axis turned by the angle of (cos, sin)[..., i]."""
    pairs = x.unflatten(-1, (-1, 2))
    a, b = pairs[..., 0], pairs[..., 1]
    return torch.stack((a * cos - b * sin, a * sin + b * cos), dim=-1).flatten(-2)


def block(x, w, cos, sin, n_heads, n_kv_heads, eps):
    """x: [B, S, d] fp64 tensor at positions 0..S-1; w: dict of fp64 tensors [out, in]."""
    B, S, d = x.shape
    G, R = n_kv_heads, n_heads // n_kv_heads          # groups and query heads per group
    D = w["wq"].shape[0] // n_heads
    xn = _rms(x, w["attn_norm"], eps)
    c, s = cos[:S, None, :], sin[:S, None, :]          # [S, 1, D/2], broadcast over heads
    q = _rotate(torch.einsum("bsi,oi->bso", xn, w["wq"]).view(B, S, n_heads, D), c, s).view(B, S, G, R, D)
    k = _rotate(torch.einsum("bsi,oi->bso", xn, w["wk"]).view(B, S, G, D), c, s)
    v = torch.einsum("bsi,oi->bso", xn, w["wv"]).view(B, S, G, D)
    logits = torch.einsum("bsgrd,btgd->bgrst", q, k) / math.sqrt(D)
    future = torch.ones(S, S, dtype=torch.bool).triu(1)  # key t after query s
    p = torch.softmax(logits.masked_fill(future, float("-inf")), dim=-1)
    o = torch.einsum("bgrst,btgd->bsgrd", p, v).reshape(B, S, n_heads * D)
    h = x + torch.einsum("bsi,oi->bso", o, w["wo"])
    hn = _rms(h, w["ffn_norm"], eps)
    gate = torch.einsum("bsi,oi->bso", hn, w["w_gate"])
    up = torch.einsum("bsi,oi->bso", hn, w["w_up"])
    act = gate * torch.sigmoid(gate) * up
    return h + torch.einsum("bsi,oi->bso", act, w["w_down"])


def model(tokens, layers, final_norm, embed, lm_head, cos, sin, n_heads, n_kv_heads, eps):
    x = embed[tokens]
    for w in layers:
        x = block(x, w, cos, sin, n_heads, n_kv_heads, eps)
    return torch.einsum("bsi,vi->bsv", _rms(x, final_norm, eps), lm_head)
