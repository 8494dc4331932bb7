"""fp64 CPU oracle of the pre-norm decoder layer (test infrastructure only).

Each function restates one definition from the pages, in their order and
notation, with numpy fp64 matmuls as the only library steps.  Nothing is
blocked, fused or reordered beyond what the definition states, so that it can
be checked against the pages by eye.

Pages cited (by title):
  [T2L]  "12 · 从 Transformer 到 LLaMA 系列"
  [CORE] "3.2 核心组件逐一拆解"
  [MOD]  "第 10 章：现代 LLaMA 架构"
  [OVW]  "深度学习进阶（三十）从 Transformer 到 LLaMA：现代 LLM 架构总览"
  [L3B]  "05 LLaMA3 Block — 从零件到发动机"

Readings taken where the pages disagree or are silent (see also the design
notes): eps inside the square root; even/odd RoPE pairs; theta_i =
base^(-2i/D); key j visible to query i iff pos_j <= pos_i; head h uses KV
group h // (H/G); SiLU on the gate projection; for bf16 layers, every
activation passed from one step to the next rounded to bf16 where it is
produced, and nowhere else.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x) -> np.ndarray:
    """Nearest-even rounding of fp64 values to the 8 significant bits of bf16.

    Used only at storage points that the configuration fixes as bf16.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2**e with 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)   # np.rint: ties to even


def linear(x, w):
    """nn.Linear without bias: y = x W^T with W in the [out, in] layout ([T2L] §八)."""
    return x @ w.T


def rms_norm(x, gamma, eps):
    """RMSNorm: gamma * x * rsqrt(mean(x^2) + eps) over the last axis.

    [T2L] §八 ``RMSNorm.forward``; [CORE] §3.2.1 ``_norm``; [MOD] §4; [OVW] §3.2.
    No mean subtraction and no bias.  eps sits inside the square root (the
    reading shared by four of the five pages).
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return gamma * (x * (1.0 / np.sqrt(ms + eps)))


def layer_norm(x, gamma, beta, eps):
    """LayerNorm: gamma * (x - mu) / sqrt(sigma^2 + eps) + beta over the last axis.

    [CORE] §3.2.1 "LayerNorm": mu is the mean over the hidden dimension and
    sigma^2 the biased variance (divided by d, not d - 1); eps sits inside the
    square root.  Not on the decoder layer's path: the pages contrast it with
    RMSNorm, which drops the centring and beta.
    """
    mu = np.mean(x, axis=-1, keepdims=True)
    var = np.mean((x - mu) ** 2, axis=-1, keepdims=True)
    return gamma * ((x - mu) / np.sqrt(var + eps)) + beta


def rope_tables(base, head_dim, max_pos):
    """cos/sin tables ``[max_pos, D/2]``: angle(p, i) = p * base^(-2i/D).

    [T2L] §八 ``RotaryEmbedding`` (inv_freq over arange(0, d, 2) / d);
    [OVW] §4.2 theta_i = base^(-2i/d).
    """
    i = np.arange(head_dim // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / head_dim)
    angle = np.outer(np.arange(max_pos, dtype=np.float64), theta)
    return np.cos(angle), np.sin(angle)


def apply_rope(x, cos, sin):
    """Rotate pairs (x[2i], x[2i+1]) by the angle whose cos/sin are given.

    [MOD] §2 (2-D rotation) and §3 ``apply_rope``: even/odd pairs of head_dim.
    ``x``: ``[..., T, D]``; ``cos``/``sin``: broadcastable to ``[..., T, D/2]``.
    """
    assert x.shape[-1] % 2 == 0, "RoPE needs an even head_dim"
    x_even = x[..., 0::2]
    x_odd = x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x_even * cos - x_odd * sin
    y[..., 1::2] = x_even * sin + x_odd * cos
    return y


def apply_rope_half(x, cos, sin):
    """Rotate pairs (x[i], x[i + D/2]) by the angle whose cos/sin are given.

    [T2L] §八 ``apply_rope``: the first and second halves of head_dim form the
    pairs, first half -> x1 cos - x2 sin, second half -> x2 cos + x1 sin, with
    the same frequency index i < D/2 as the even/odd form.
    """
    assert x.shape[-1] % 2 == 0, "RoPE needs an even head_dim"
    half = x.shape[-1] // 2
    x1 = x[..., :half]
    x2 = x[..., half:]
    y = np.empty_like(x)
    y[..., :half] = x1 * cos - x2 * sin
    y[..., half:] = x2 * cos + x1 * sin
    return y


ROPE_STYLES = {"even_odd": apply_rope, "half": apply_rope_half}


def silu(z):
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)).  [T2L] §5.1; [CORE] §3.2.2."""
    return z / (1.0 + np.exp(-z))


def _keep(a):
    return a


def swiglu_mlp(x, w_gate, w_up, w_down, store=_keep):
    """SwiGLU MLP: down(SiLU(x W_gate^T) * (x W_up^T)), no bias.

    [CORE] §3.2.2 ``SwiGLUFFN``; [L3B] §4.1 ``LlamaMLP`` and §6 (the SiLU goes on
    the gate projection, not on up); [MOD] §5.  ``store`` is applied to the gated
    product, the activation handed to the down projection.
    """
    return store(silu(x @ w_gate.T) * (x @ w_up.T)) @ w_down.T


def attention(q, k, v, q_pos, k_len):
    """Causal grouped-query scaled dot-product attention.

    ``q``: ``[B, H, S, D]`` at absolute positions ``q_pos`` ``[B, S]``;
    ``k``, ``v``: ``[B, G, T, D]``, key slot j holding absolute position j, of
    which the first ``k_len[b]`` are valid.  Query head h reads KV group
    h // (H/G) ([T2L] §八 ``repeat_interleave`` on dim 1; [MOD] §6
    ``repeat_kv``).  Scores are q.k / sqrt(D) ([OVW] §1.1); key j is visible
    to query i iff j <= pos_i ([T2L] §八 ``is_causal=True``; [MOD] §7 decode
    mask over past_len + 1 keys).  Returns ``[B, H, S, D]``.
    """
    B, H, S, D = q.shape
    G = k.shape[1]
    assert H % G == 0, "n_heads must be a multiple of n_kv_heads"
    rep = H // G
    out = np.empty_like(q)
    for b in range(B):
        T = int(k_len[b])
        allowed = np.arange(T)[None, :] <= np.asarray(q_pos[b])[:, None]      # [S, T]
        for h in range(H):
            g = h // rep
            scores = (q[b, h] @ k[b, g, :T].T) / np.sqrt(D)
            scores = np.where(allowed, scores, -np.inf)
            scores = scores - scores.max(axis=-1, keepdims=True)
            p = np.exp(scores)
            p = p / p.sum(axis=-1, keepdims=True)
            out[b, h] = p @ v[b, g, :T]
    return out


def decoder_layer(x, w, cos, sin, *, n_heads, n_kv_heads, head_dim, rms_eps,
                  past_k=None, past_v=None, past_len=None, store_bf16=False, rope="even_odd"):
    """One pre-norm decoder layer, prefill or incremental.

    [L3B] §3.1 and §4.2 (save residual, norm, sublayer, add back, twice, with
    two separate norms ``input_layernorm``/``post_attention_layernorm``);
    [MOD] §9 ``llama_block(x, position_ids, past_kv)``; [T2L] §八 ``LlamaBlock``.

    ``x``: ``[B, S, d]``; ``w``: dict of fp64 arrays in ``nn.Linear`` layout
    (``wq [H*D, d]`` ...).  New tokens of sequence b sit at positions
    ``past_len[b] + s`` ([MOD] §3: position_id = past_len); ``past_k/v``
    ``[B, G, T, D]`` hold the cache, slots ``[0, past_len[b])`` valid.

    ``store_bf16``: the layer keeps its activations in bf16 (the configurations'
    "bf16 weights and activations, fp32 accumulation").  Every tensor handed from
    one step of the layer to the next is then rounded to bf16 once, where it is
    produced: the normed input, q and k after RoPE, v (the cache), the attention
    output, h, the normed h and the gated MLP activation.  Arithmetic inside a step
    stays exact.
    ``rope``: "even_odd" ([MOD] §3, the default) or "half" ([T2L] §八) pairing.
    Returns ``(out [B,S,d], k_new [B,G,S,D], v_new [B,G,S,D])``.
    """
    st = round_bf16 if store_bf16 else _keep
    B, S, d = x.shape
    H, G, D = n_heads, n_kv_heads, head_dim
    if past_len is None:
        past_len = np.zeros(B, dtype=np.int64)
    past_len = np.asarray(past_len, dtype=np.int64)
    pos = past_len[:, None] + np.arange(S)[None, :]                     # [B, S]

    # attention half
    residual = x
    xn = st(rms_norm(x, w["attn_norm"], rms_eps))
    q = (xn @ w["wq"].T).reshape(B, S, H, D).transpose(0, 2, 1, 3)       # [B, H, S, D]
    k = (xn @ w["wk"].T).reshape(B, S, G, D).transpose(0, 2, 1, 3)       # [B, G, S, D]
    v = (xn @ w["wv"].T).reshape(B, S, G, D).transpose(0, 2, 1, 3)
    c = cos[pos][:, None, :, :]                                          # [B, 1, S, D/2]
    s = sin[pos][:, None, :, :]
    rot = ROPE_STYLES[rope]
    q = st(rot(q, c, s))                                                 # RoPE on q and k only
    k = st(rot(k, c, s))
    v = st(v)

    # keys of sequence b: cached slots [0, past_len[b]) then the S new ones
    T = int((past_len + S).max())
    kk = np.zeros((B, G, T, D))
    vv = np.zeros((B, G, T, D))
    for b in range(B):
        P = int(past_len[b])
        if P:
            kk[b, :, :P] = past_k[b, :, :P]
            vv[b, :, :P] = past_v[b, :, :P]
        kk[b, :, P:P + S] = k[b]
        vv[b, :, P:P + S] = v[b]
    o = st(attention(q, kk, vv, pos, past_len + S))                       # [B, H, S, D]
    o = o.transpose(0, 2, 1, 3).reshape(B, S, H * D)
    h = st(residual + o @ w["wo"].T)

    # MLP half
    residual = h
    hn = st(rms_norm(h, w["ffn_norm"], rms_eps))
    out = residual + swiglu_mlp(hn, w["w_gate"], w["w_up"], w["w_down"], store=st)
    return out, k, v


def stack_forward(tokens, layers, final_norm, embed, lm_head, cos, sin, *, n_heads,
                  n_kv_heads, head_dim, rms_eps, store_bf16=False, rope="even_odd"):
    """embed -> layers -> final RMSNorm -> untied LM head ([T2L] §八 ``LlamaModel.forward``).

    ``layers`` yields one weight dict per layer (so callers can stream them).
    With ``store_bf16`` the activations are bf16 (see ``decoder_layer``): each
    layer's output and the final normed activation are rounded once too.
    Returns logits ``[B, S, V]``.
    """
    x = embed[tokens]
    for w in layers:
        x, _, _ = decoder_layer(x, w, cos, sin, n_heads=n_heads, n_kv_heads=n_kv_heads,
                                head_dim=head_dim, rms_eps=rms_eps, store_bf16=store_bf16, rope=rope)
        if store_bf16:
            x = round_bf16(x)
    xn = rms_norm(x, final_norm, rms_eps)                                 # the final norm Pre-LN needs
    if store_bf16:
        xn = round_bf16(xn)
    return xn @ lm_head.T


def stack_decode(tokens, positions, layers, caches, final_norm, embed, lm_head, cos, sin, *, n_heads,
                 n_kv_heads, head_dim, rms_eps, store_bf16=False, rope="even_odd"):
    """One autoregressive step of the whole model for B sequences.

    [MOD] §7 decode (one new token per sequence at position_id = past_len,
    its K/V appended to each layer's cache) through every layer, then the final
    RMSNorm and the untied LM head of [T2L] §八 ``LlamaModel.forward``.
    ``tokens``, ``positions``: ``[B]``; ``caches``: one ``(k, v)`` pair
    ``[B, G, T, D]`` per layer, slots ``[0, positions[b])`` valid.  Returns the
    logits ``[B, V]`` and, per layer, the new token's ``(k, v)`` ``[B, G, 1, D]``.
    """
    positions = np.asarray(positions, dtype=np.int64)
    x = embed[np.asarray(tokens)][:, None, :]                              # [B, 1, d]
    new_kv = []
    for w, (pk, pv) in zip(layers, caches):
        x, k, v = decoder_layer(x, w, cos, sin, n_heads=n_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
                                rms_eps=rms_eps, past_k=pk, past_v=pv, past_len=positions,
                                store_bf16=store_bf16, rope=rope)
        if store_bf16:
            x = round_bf16(x)
        new_kv.append((k, v))
    xn = rms_norm(x[:, 0], final_norm, rms_eps)
    if store_bf16:
        xn = round_bf16(xn)
    return xn @ lm_head.T, new_kv


def param_count(vocab, d, n_layers, n_heads, n_kv_heads, d_inter, tied=False):
    """Parameters of the model of [T2L] §八: embedding, layers, final norm, LM head.

    Per layer: wq [H*D, d], wk/wv [G*D, d], wo [d, H*D], the three SwiGLU
    matrices (3 * d * d_inter, [CORE] §3.2.2) and two RMSNorm gammas [d].
    """
    D = d // n_heads
    attn = d * n_heads * D + 2 * d * n_kv_heads * D + n_heads * D * d
    mlp = 3 * d * d_inter
    norms = 2 * d
    head = 0 if tied else vocab * d
    return vocab * d + n_layers * (attn + mlp + norms) + d + head


def kv_cache_bytes(n_layers, B, n_kv_heads, T, head_dim, bytes_per_elem=2):
    """K and V caches of ``[L, B, G, T, D]`` elements each ([MOD] §6 and §8)."""
    return 2 * n_layers * B * n_kv_heads * T * head_dim * bytes_per_elem
