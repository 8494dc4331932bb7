"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: numbers the
pages print (tests/golden), closed forms, invariants, special cases that reduce to a
library routine, and brute force on tiny inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden
from llama_decoder_block_gb300 import synth
import torch_block

RNG = np.random.default_rng(12345)


def _layer_w(d, H, G, D, I, gamma_noise=0.1, std=0.02, rng=RNG):
    w = {
        "attn_norm": 1 + gamma_noise * rng.standard_normal(d),
        "ffn_norm": 1 + gamma_noise * rng.standard_normal(d),
        "wq": std * rng.standard_normal((H * D, d)), "wk": std * rng.standard_normal((G * D, d)),
        "wv": std * rng.standard_normal((G * D, d)), "wo": std * rng.standard_normal((d, H * D)),
        "w_gate": std * rng.standard_normal((I, d)), "w_up": std * rng.standard_normal((I, d)),
        "w_down": std * rng.standard_normal((d, I)),
    }
    return w


# ------------------------------------------------------------------ bf16 storage rounding

def test_round_bf16_matches_independent_bit_rounding():
    # the oracle rounds fp64 via frexp; the input generator rounds fp32 bit patterns.
    x = np.concatenate([RNG.standard_normal(200000) * s for s in (1e-3, 1.0, 1e3)]).astype(np.float32)
    a = oracle.round_bf16(x.astype(np.float64))
    b = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x)).astype(np.float64)
    assert np.array_equal(a, b)


def test_round_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even significand wins (1.0);
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    assert oracle.round_bf16(1 + 2.0 ** -8) == 1.0
    assert oracle.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert oracle.round_bf16(-(1 + 2.0 ** -8)) == -1.0
    assert oracle.round_bf16(0.0) == 0.0


# ------------------------------------------------------------------ linear

def test_linear_uses_out_in_layout():
    # W = [[1, 2], [3, 4], [5, 6]] maps 2 inputs to 3 outputs: y_j = sum_i W[j, i] x_i
    y = oracle.linear(np.array([[1.0, -1.0]]), np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]]))
    assert np.array_equal(y, [[-1.0, -1.0, -1.0]])
    y = oracle.linear(np.array([[2.0, 0.5]]), np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]]))
    assert np.array_equal(y, [[3.0, 8.0, 13.0]])


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_worked_example():
    g = golden("rmsnorm_worked_example.txt")
    x = np.array(g["x"])
    y = oracle.rms_norm(x, np.ones(2), 0.0)
    dec = int(g["decimals"][0])
    assert np.array_equal(np.round(y, dec), np.array(g["y"]))
    assert round(float(x[0] / y[0]), dec) == g["rms"][0]


def test_rmsnorm_output_rms_closed_form():
    # gamma = 1: rms(y) = sqrt(ms / (ms + eps)) exactly, i.e. 1 within eps / (2 ms).
    x = RNG.standard_normal((7, 513))
    for eps in (1e-6, 1e-5, 0.3):
        y = oracle.rms_norm(x, np.ones(513), eps)
        ms = np.mean(x * x, axis=-1)
        assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), np.sqrt(ms / (ms + eps)), rtol=1e-14, atol=0)


def test_rmsnorm_eps_inside_the_square_root():
    # x = [3, 4], eps = 1: rsqrt(12.5 + 1) = 1/sqrt(13.5); the other printed form
    # x / (RMS(x) + eps) would give x / (sqrt(12.5) + 1).
    y = oracle.rms_norm(np.array([3.0, 4.0]), np.ones(2), 1.0)
    assert np.allclose(y, np.array([3.0, 4.0]) / math.sqrt(13.5), rtol=1e-15)
    assert not np.allclose(y, np.array([3.0, 4.0]) / (math.sqrt(12.5) + 1.0), rtol=1e-6)


def test_rmsnorm_gamma_scales_after_normalising():
    x = RNG.standard_normal((3, 64))
    g = RNG.standard_normal(64)
    assert np.allclose(oracle.rms_norm(x, g, 1e-5), g * oracle.rms_norm(x, np.ones(64), 1e-5), rtol=1e-14)
    # scale invariance: RMSNorm(c x) = RMSNorm(x) for c > 0 when eps = 0
    assert np.allclose(oracle.rms_norm(5.5 * x, g, 0.0), oracle.rms_norm(x, g, 0.0), rtol=1e-13)


def test_rmsnorm_statistics_of_normal_input():
    # page "深度学习进阶（三十）..." §3.2: output mean ~0 and std ~1 for x ~ N(0,1), gamma = 1
    x = RNG.standard_normal((2, 10, 512))
    y = oracle.rms_norm(x, np.ones(512), 1e-6)
    assert abs(y.mean()) < 0.03 and abs(y.std() - 1) < 0.03


# ------------------------------------------------------------------ LayerNorm

def test_layernorm_two_element_closed_form():
    # "3.2 核心组件逐一拆解" §3.2.1: x = [1, 3] has mean 2 and biased variance 1, so with
    # eps = 0 the output is [-1, 1]; with eps = 3, [-1, 1] / sqrt(1 + 3) = [-0.5, 0.5].
    one, zero = np.ones(2), np.zeros(2)
    assert np.array_equal(oracle.layer_norm(np.array([1.0, 3.0]), one, zero, 0.0), [-1.0, 1.0])
    assert np.array_equal(oracle.layer_norm(np.array([1.0, 3.0]), one, zero, 3.0), [-0.5, 0.5])
    # gamma scales the normalised value, beta is added after it
    y = oracle.layer_norm(np.array([1.0, 3.0]), np.array([2.0, -4.0]), np.array([0.25, 0.5]), 0.0)
    assert np.array_equal(y, [-1.75, -3.5])


def test_layernorm_output_moments_closed_form():
    # gamma = 1, beta = 0: each row has mean 0 and variance var / (var + eps) exactly.
    x = 3.0 + 2.0 * RNG.standard_normal((6, 1000))
    for eps in (1e-5, 0.5):
        y = oracle.layer_norm(x, np.ones(1000), np.zeros(1000), eps)
        var = np.var(x, axis=-1)
        assert np.allclose(y.mean(-1), 0.0, atol=1e-13)
        assert np.allclose(np.mean(y * y, axis=-1), var / (var + eps), rtol=1e-13, atol=0)


def test_layernorm_shift_and_scale_invariance():
    # re-centring removes any constant shift; with eps = 0 a positive scale cancels too
    x = RNG.standard_normal((4, 96))
    g, b = RNG.standard_normal(96), RNG.standard_normal(96)
    base = oracle.layer_norm(x, g, b, 1e-5)
    assert np.allclose(oracle.layer_norm(x + 7.25, g, b, 1e-5), base, rtol=1e-11, atol=1e-12)
    assert np.allclose(oracle.layer_norm(3.0 * x, g, b, 0.0), oracle.layer_norm(x, g, b, 0.0), rtol=1e-12,
                       atol=1e-13)


def test_layernorm_is_rmsnorm_of_the_centred_row_plus_beta():
    # the biased variance is the mean square of x - mu, so LN(x) = RMSNorm(x - mu) + beta
    x = RNG.standard_normal((5, 128)) + 0.7
    g, b = RNG.standard_normal(128), RNG.standard_normal(128)
    centred = x - x.mean(-1, keepdims=True)
    assert np.allclose(oracle.layer_norm(x, g, b, 1e-5), oracle.rms_norm(centred, g, 1e-5) + b, rtol=1e-12,
                       atol=1e-13)


def test_layernorm_matches_torch_layer_norm_in_fp64():
    x = RNG.standard_normal((9, 257))
    g, b = RNG.standard_normal(257), RNG.standard_normal(257)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (257,), torch.from_numpy(g), torch.from_numpy(b),
                                         1e-5).numpy()
    assert np.allclose(oracle.layer_norm(x, g, b, 1e-5), ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ RoPE

def test_rope_special_frequencies():
    # theta_0 = 1 (angle = p); for D = 128 and base = 1e4, theta_32 = 1e4^(-1/2) = 0.01.
    cos, sin = oracle.rope_tables(1e4, 128, 301)
    p = np.arange(301)
    assert np.allclose(cos[:, 0], np.cos(p), atol=1e-15) and np.allclose(sin[:, 0], np.sin(p), atol=1e-15)
    assert abs(cos[100, 32] - math.cos(1.0)) < 1e-14 and abs(sin[100, 32] - math.sin(1.0)) < 1e-14
    assert abs(cos[300, 64 - 1] - math.cos(300 * 1e4 ** (-126 / 128))) < 1e-15


def test_rope_pairs_are_even_odd():
    # a one-hot on coordinate 0 rotates inside the pair (0, 1), not (0, D/2).
    D = 8
    cos, sin = oracle.rope_tables(1e4, D, 5)
    e0 = np.zeros(D)
    e0[0] = 1
    y = oracle.apply_rope(e0[None, :], cos[3:4], sin[3:4])[0]
    assert np.allclose(y, [math.cos(3), math.sin(3), 0, 0, 0, 0, 0, 0], atol=1e-15)
    e3 = np.zeros(D)
    e3[3] = 1     # odd member of pair i = 1, theta_1 = 1e4^(-2/8)
    a = 2 * 1e4 ** (-0.25)
    y = oracle.apply_rope(e3[None, :], cos[2:3], sin[2:3])[0]
    assert np.allclose(y, [0, 0, -math.sin(a), math.cos(a), 0, 0, 0, 0], atol=1e-15)


def test_rope_two_dim_rotation_formula():
    # page "第 10 章" §2: [x1, x2] -> [x1 cos t - x2 sin t, x1 sin t + x2 cos t]; D = 2 has theta = 1
    cos, sin = oracle.rope_tables(10.0, 2, 7)
    x = np.array([[0.3, -1.7]])
    for p in range(7):
        y = oracle.apply_rope(x, cos[p:p + 1], sin[p:p + 1])[0]
        assert np.allclose(y, [0.3 * math.cos(p) + 1.7 * math.sin(p), 0.3 * math.sin(p) - 1.7 * math.cos(p)],
                           atol=1e-15)


def test_rope_preserves_norm_and_position_zero_is_identity():
    cos, sin = oracle.rope_tables(5e5, 128, 4096)
    x = RNG.standard_normal((4096, 128))
    y = oracle.apply_rope(x, cos, sin)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    assert np.array_equal(y[0], x[0])


def test_rope_scores_depend_only_on_offset():
    cos, sin = oracle.rope_tables(1e4, 64, 600)
    q = RNG.standard_normal(64)
    k = RNG.standard_normal(64)
    for m, n, s in ((5, 2, 100), (17, 17, 400), (3, 250, 77)):
        a = oracle.apply_rope(q[None], cos[m:m + 1], sin[m:m + 1]) @ oracle.apply_rope(k[None], cos[n:n + 1], sin[n:n + 1]).T
        b = oracle.apply_rope(q[None], cos[m + s:m + s + 1], sin[m + s:m + s + 1]) @ \
            oracle.apply_rope(k[None], cos[n + s:n + s + 1], sin[n + s:n + s + 1]).T
        assert abs(a.item() - b.item()) < 1e-12


def test_rope_half_pairs_coordinate_i_with_i_plus_half():
    # "12 · 从 Transformer 到 LLaMA 系列" §八 apply_rope: a one-hot on coordinate 0 rotates into
    # coordinate D/2 (not 1); on coordinate D/2 + 1 it rotates back into coordinate 1 with
    # theta_1 = base^(-2/D).
    D = 8
    cos, sin = oracle.rope_tables(1e4, D, 5)
    e0 = np.zeros(D)
    e0[0] = 1
    y = oracle.apply_rope_half(e0[None, :], cos[3:4], sin[3:4])[0]
    assert np.allclose(y, [math.cos(3), 0, 0, 0, math.sin(3), 0, 0, 0], atol=1e-15)
    e5 = np.zeros(D)
    e5[5] = 1
    a = 2 * 1e4 ** (-0.25)
    y = oracle.apply_rope_half(e5[None, :], cos[2:3], sin[2:3])[0]
    assert np.allclose(y, [0, -math.sin(a), 0, 0, 0, math.cos(a), 0, 0], atol=1e-15)


def test_rope_half_is_even_odd_on_interleaved_coordinates():
    # moving coordinate i to 2i and i + D/2 to 2i + 1 turns one pairing into the other
    D = 64
    cos, sin = oracle.rope_tables(1e4, D, 50)
    x = RNG.standard_normal((50, D))
    perm = np.empty(D, dtype=int)
    perm[0::2] = np.arange(D // 2)
    perm[1::2] = np.arange(D // 2) + D // 2
    y_half = oracle.apply_rope_half(x, cos, sin)
    y_eo = oracle.apply_rope(x[:, perm], cos, sin)
    assert np.allclose(y_half[:, perm], y_eo, rtol=0, atol=1e-14)


def test_rope_half_preserves_norm_and_relative_position():
    cos, sin = oracle.rope_tables(1e4, 64, 600)
    x = RNG.standard_normal((600, 64))
    y = oracle.apply_rope_half(x, cos, sin)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    assert np.array_equal(y[0], x[0])
    q, k = RNG.standard_normal(64), RNG.standard_normal(64)
    r = lambda v, m: oracle.apply_rope_half(v[None], cos[m:m + 1], sin[m:m + 1])
    for m, n, s in ((5, 2, 100), (3, 250, 77)):
        assert abs((r(q, m) @ r(k, n).T).item() - (r(q, m + s) @ r(k, n + s).T).item()) < 1e-12


def test_layer_with_half_rope_equals_even_odd_layer_with_permuted_projections():
    # permuting the rows of Wq and Wk inside each head by the interleaving map leaves every
    # attention score, and so the layer output, unchanged
    d, H, G, D, I = 64, 4, 2, 16, 96
    w = _layer_w(d, H, G, D, I)
    perm = np.empty(D, dtype=int)
    perm[0::2] = np.arange(D // 2)
    perm[1::2] = np.arange(D // 2) + D // 2
    wp = dict(w)
    wp["wq"] = w["wq"].reshape(H, D, d)[:, perm].reshape(H * D, d)
    wp["wk"] = w["wk"].reshape(G, D, d)[:, perm].reshape(G * D, d)
    cos, sin = oracle.rope_tables(1e4, D, 40)
    x = RNG.standard_normal((2, 40, d))
    kw = dict(n_heads=H, n_kv_heads=G, head_dim=D, rms_eps=1e-5)
    out_h, k_h, _ = oracle.decoder_layer(x, w, cos, sin, rope="half", **kw)
    out_e, k_e, _ = oracle.decoder_layer(x, wp, cos, sin, rope="even_odd", **kw)
    assert np.allclose(out_h, out_e, rtol=1e-12, atol=1e-12)
    assert np.allclose(k_h[..., perm], k_e, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ attention

def _attn_case(B, H, G, S, D, rng=RNG):
    q = rng.standard_normal((B, H, S, D))
    k = rng.standard_normal((B, G, S, D))
    v = rng.standard_normal((B, G, S, D))
    pos = np.tile(np.arange(S), (B, 1))
    return q, k, v, pos, np.full(B, S)


@pytest.mark.parametrize("H,G", [(4, 4), (8, 2), (6, 1)])
def test_attention_matches_library_sdpa(H, G):
    q, k, v, pos, kl = _attn_case(2, H, G, 37, 16)
    ours = oracle.attention(q, k, v, pos, kl)
    rep = H // G
    t = lambda a: torch.from_numpy(a)
    ref = torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k).repeat_interleave(rep, dim=1), t(v).repeat_interleave(rep, dim=1), is_causal=True)
    assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_on_repeated_kv():
    q, k, v, pos, kl = _attn_case(1, 8, 2, 20, 8)
    gqa = oracle.attention(q, k, v, pos, kl)
    mha = oracle.attention(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), pos, kl)
    assert np.allclose(gqa, mha, rtol=0, atol=1e-15)
    # head h reads group h // (H/G): heads 0..3 see group 0 only
    k2, v2 = k.copy(), v.copy()
    k2[:, 1] += 1.0
    v2[:, 1] += 1.0
    gqa2 = oracle.attention(q, k2, v2, pos, kl)
    assert np.array_equal(gqa[:, :4], gqa2[:, :4]) and not np.allclose(gqa[:, 4:], gqa2[:, 4:])


def test_causal_boundary_is_inclusive():
    # q = 0 gives equal scores, so row i averages the visible V rows; with V = one-hot(j)
    # rows, O[i, j] = 1/(i+1) for j <= i and 0 beyond.
    S = 12
    q = np.zeros((1, 1, S, S))
    k = RNG.standard_normal((1, 1, S, S))
    v = np.eye(S)[None, None]
    o = oracle.attention(q, k, v, np.arange(S)[None], np.array([S]))[0, 0]
    expect = np.tril(np.ones((S, S))) / np.arange(1, S + 1)[:, None]
    assert np.allclose(o, expect, rtol=0, atol=1e-15)


def test_decode_mask_sees_the_whole_cache():
    # one query at position p sees slots 0..p: p + 1 keys, not only itself
    p = 9
    q = np.zeros((1, 2, 1, 4))
    k = RNG.standard_normal((1, 1, 16, 4))
    v = np.tile(np.arange(16.0)[:, None], (1, 4))[None, None]
    o = oracle.attention(q, k, v, np.array([[p]]), np.array([16]))
    assert np.allclose(o, np.mean(np.arange(p + 1.0)), atol=1e-14)


# ------------------------------------------------------------------ SwiGLU

def test_silu_closed_forms():
    z = RNG.standard_normal(1000) * 6
    assert np.allclose(oracle.silu(z) - oracle.silu(-z), z, rtol=1e-14, atol=1e-14)
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-15 and abs(oracle.silu(-40.0)) < 1e-15


def test_swiglu_gate_example():
    g = golden("swiglu_gate_example.txt")
    gate_signal, up = np.array(g["gate"]), np.array(g["up"])
    # pre-activations whose SiLU is the printed gate signal (bisection on the monotone branch)
    pre = []
    for target in gate_signal:
        lo, hi = -1e-9 if target == 0 else 0.0, 10.0
        for _ in range(200):
            mid = 0.5 * (lo + hi)
            lo, hi = (mid, hi) if oracle.silu(mid) < target else (lo, mid)
        pre.append(0.5 * (lo + hi))
    out = oracle.swiglu_mlp(np.ones((1, 3)), np.diag(pre), np.diag(up), np.eye(3))[0]
    assert np.allclose(out, g["after"], atol=1e-12)


def test_swiglu_activation_is_on_gate_not_up():
    x = np.ones((1, 1))
    out = oracle.swiglu_mlp(x, np.array([[-50.0]]), np.array([[3.0]]), np.array([[1.0]]))
    assert abs(out.item()) < 1e-18       # SiLU(-50) * 3; swapped it would be SiLU(3) * -50


def test_param_counts_printed_on_the_page():
    g = golden("param_counts.txt")
    kw = dict(vocab=int(g["vocab"][0]), d=int(g["d"][0]), n_layers=int(g["n_layers"][0]),
              n_heads=int(g["n_heads"][0]), d_inter=int(g["d_inter"][0]))
    gqa = oracle.param_count(n_kv_heads=int(g["gqa_kv_heads"][0]), **kw)
    mha = oracle.param_count(n_kv_heads=int(g["mha_kv_heads"][0]), **kw)
    assert gqa == int(g["gqa_total"][0]) and mha == int(g["mha_total"][0])
    assert mha - gqa == int(g["saved"][0])
    # the SwiGLU share: 3 * d * d_inter per layer
    d, I = kw["d"], kw["d_inter"]
    assert oracle.param_count(**{**kw, "d_inter": I + 1}, n_kv_heads=2) - gqa == kw["n_layers"] * 3 * d


def test_kv_cache_bytes_printed_on_the_page():
    g = golden("kv_cache_bytes.txt")
    args = [int(g[k][0]) for k in ("layers", "B", "G", "T", "D", "bytes_per_elem")]
    assert oracle.kv_cache_bytes(*args) == int(g["gqa_bytes"][0])
    args[2] = int(g["H"][0])
    assert oracle.kv_cache_bytes(*args) == int(g["mha_over_gqa"][0]) * int(g["gqa_bytes"][0])


# ------------------------------------------------------------------ the layer

def _tiny_layer_inputs():
    wl = synth.WORKLOADS["tiny_f32_b1_s16"]
    L = wl.layer
    w = {k: v.f64() for k, v in synth.layer_weights(wl).items()}
    x = synth.activations(wl).f64()
    cos, sin = oracle.rope_tables(L.rope_base, L.head_dim, 64)
    cos, sin = cos.astype(np.float32).astype(np.float64), sin.astype(np.float32).astype(np.float64)
    kw = dict(n_heads=L.n_heads, n_kv_heads=L.n_kv_heads, head_dim=L.head_dim, rms_eps=L.rms_eps)
    return wl, w, x, cos, sin, kw


def test_layer_brute_force_tiny_config_against_torch_statement():
    wl, w, x, cos, sin, kw = _tiny_layer_inputs()
    ours, _, _ = oracle.decoder_layer(x, w, cos, sin, **kw)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    ref = torch_block.block(t(x), {k: t(v) for k, v in w.items()}, t(cos), t(sin),
                            kw["n_heads"], kw["n_kv_heads"], kw["rms_eps"])
    assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_layer_brute_force_bigger_random_gqa():
    rng = np.random.default_rng(7)
    B, S, d, H, G, D, I = 2, 45, 96, 6, 3, 16, 160
    w = _layer_w(d, H, G, D, I, std=0.1, rng=rng)
    x = rng.standard_normal((B, S, d))
    cos, sin = oracle.rope_tables(500000.0, D, 64)
    kw = dict(n_heads=H, n_kv_heads=G, head_dim=D, rms_eps=1e-5)
    ours, _, _ = oracle.decoder_layer(x, w, cos, sin, **kw)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    ref = torch_block.block(t(x), {k: t(v) for k, v in w.items()}, t(cos), t(sin), H, G, 1e-5)
    assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_layer_zero_weights_is_identity_and_norms_are_separate():
    rng = np.random.default_rng(3)
    d, H, G, D, I = 32, 4, 2, 8, 48
    w = _layer_w(d, H, G, D, I, std=0.2, rng=rng)
    x = rng.standard_normal((1, 9, d))
    cos, sin = oracle.rope_tables(1e4, D, 16)
    kw = dict(n_heads=H, n_kv_heads=G, head_dim=D, rms_eps=1e-5)
    z = {k: (np.zeros_like(v) if k.startswith("w") else v) for k, v in w.items()}
    assert np.array_equal(oracle.decoder_layer(x, z, cos, sin, **kw)[0], x)
    w2 = dict(w)
    w2["ffn_norm"] = w["ffn_norm"] * 3.0
    assert not np.allclose(oracle.decoder_layer(x, w2, cos, sin, **kw)[0], oracle.decoder_layer(x, w, cos, sin, **kw)[0])


def test_layer_causality():
    rng = np.random.default_rng(11)
    d, H, G, D, I = 64, 4, 2, 16, 96
    w = _layer_w(d, H, G, D, I, std=0.1, rng=rng)
    x = rng.standard_normal((2, 24, d))
    cos, sin = oracle.rope_tables(1e4, D, 32)
    kw = dict(n_heads=H, n_kv_heads=G, head_dim=D, rms_eps=1e-5)
    base, _, _ = oracle.decoder_layer(x, w, cos, sin, **kw)
    t = 13
    x2 = x.copy()
    x2[:, t + 1:] = rng.standard_normal(x2[:, t + 1:].shape) * 5
    pert, _, _ = oracle.decoder_layer(x2, w, cos, sin, **kw)
    assert np.allclose(pert[:, :t + 1], base[:, :t + 1], rtol=0, atol=1e-13)
    assert not np.allclose(pert[:, t + 1:], base[:, t + 1:])
    # prefix truncation: an S'-token run equals the first S' rows of the S-token run
    short, _, _ = oracle.decoder_layer(x[:, :t + 1], w, cos, sin, **kw)
    assert np.allclose(short, base[:, :t + 1], rtol=0, atol=1e-13)


@pytest.mark.parametrize("store_bf16", [False, True])
def test_kv_cache_decode_equals_full_prefill_row(store_bf16):
    rng = np.random.default_rng(5)
    d, H, G, D, I = 64, 8, 2, 16, 96
    w = _layer_w(d, H, G, D, I, std=0.1, rng=rng)
    B, S = 3, 20
    x = rng.standard_normal((B, S, d))
    cos, sin = oracle.rope_tables(1e4, D, 64)
    kw = dict(n_heads=H, n_kv_heads=G, head_dim=D, rms_eps=1e-6, store_bf16=store_bf16)
    full, kf, vf = oracle.decoder_layer(x, w, cos, sin, **kw)
    # per-sequence cached lengths; cache holds the full run's K/V, slots >= t unused
    t = np.array([7, 19, 0])
    cache_k = np.full((B, G, 32, D), np.nan)
    cache_v = np.full((B, G, 32, D), np.nan)
    cache_k[:, :, :S] = kf
    cache_v[:, :, :S] = vf
    xs = x[np.arange(B), t][:, None, :]
    dec, kd, vd = oracle.decoder_layer(xs, w, cos, sin, past_k=cache_k, past_v=cache_v, past_len=t, **kw)
    assert np.allclose(dec[:, 0], full[np.arange(B), t], rtol=0, atol=1e-12)
    assert np.allclose(kd[:, :, 0], kf[np.arange(B), :, t], rtol=0, atol=1e-12)
    # chunked: the second half on top of the first half's cache equals the full run
    h1, k1, v1 = oracle.decoder_layer(x[:, :11], w, cos, sin, **kw)
    h2, _, _ = oracle.decoder_layer(x[:, 11:], w, cos, sin, past_k=k1, past_v=v1, past_len=np.full(B, 11), **kw)
    assert np.allclose(np.concatenate([h1, h2], axis=1), full, rtol=0, atol=1e-12)
    # per-sequence starts: sequence b's 6-token chunk sits on its own cached length t2[b]
    # (the cache is the full run's, slots >= t2[b] poisoned) and equals rows t2[b]..t2[b]+5
    t2 = np.array([3, 14, 9])
    ck = np.full((B, G, 32, D), np.nan)
    cv = np.full((B, G, 32, D), np.nan)
    for b in range(B):
        ck[b, :, :t2[b]] = kf[b, :, :t2[b]]
        cv[b, :, :t2[b]] = vf[b, :, :t2[b]]
    xc = np.stack([x[b, t2[b]:t2[b] + 6] for b in range(B)])
    hc, kc, _ = oracle.decoder_layer(xc, w, cos, sin, past_k=ck, past_v=cv, past_len=t2, **kw)
    for b in range(B):
        assert np.allclose(hc[b], full[b, t2[b]:t2[b] + 6], rtol=0, atol=1e-12)
        assert np.allclose(kc[b], kf[b, :, t2[b]:t2[b] + 6], rtol=0, atol=1e-12)


def test_stack_brute_force_against_torch_statement():
    rng = np.random.default_rng(9)
    V, d, H, G, D, I, S, n = 50, 32, 4, 2, 8, 48, 10, 3
    layers = [_layer_w(d, H, G, D, I, std=0.2, rng=rng) for _ in range(n)]
    embed = 0.5 * rng.standard_normal((V, d))
    lm = 0.2 * rng.standard_normal((V, d))
    fn = 1 + 0.1 * rng.standard_normal(d)
    tokens = rng.integers(0, V, size=(2, S))
    cos, sin = oracle.rope_tables(1e4, D, 16)
    ours = oracle.stack_forward(tokens, layers, fn, embed, lm, cos, sin, n_heads=H, n_kv_heads=G,
                                head_dim=D, rms_eps=1e-5)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    ref = torch_block.model(t(tokens), [{k: t(v) for k, v in w.items()} for w in layers], t(fn), t(embed),
                            t(lm), t(cos), t(sin), H, G, 1e-5)
    assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("store_bf16", [False, True])
def test_stack_decode_equals_full_forward_last_row(store_bf16):
    # "第 10 章：现代 LLaMA 架构" §7, the KV-cache check: the logits of full_forward(prompt +
    # next_token) at the last position equal those of prefill(prompt) followed by
    # decode_one(next_token, past_kv).  Prompt lengths differ per sequence.
    rng = np.random.default_rng(21)
    V, d, H, G, D, I, S, n = 40, 32, 4, 2, 8, 48, 12, 3
    layers = [_layer_w(d, H, G, D, I, std=0.2, rng=rng) for _ in range(n)]
    embed = 0.5 * rng.standard_normal((V, d))
    lm = 0.2 * rng.standard_normal((V, d))
    fn = 1 + 0.1 * rng.standard_normal(d)
    tokens = rng.integers(0, V, size=(3, S))
    cos, sin = oracle.rope_tables(1e4, D, 16)
    kw = dict(n_heads=H, n_kv_heads=G, head_dim=D, rms_eps=1e-5, store_bf16=store_bf16)
    full = oracle.stack_forward(tokens, layers, fn, embed, lm, cos, sin, **kw)
    # prefill: every layer's K/V of the whole prompt; slots at or past each prompt's end are NaN
    t = np.array([5, 11, 0])
    caches, x = [], embed[tokens]
    for w in layers:
        x, k, v = oracle.decoder_layer(x, w, cos, sin, **kw)
        if store_bf16:
            x = oracle.round_bf16(x)
        k, v = k.copy(), v.copy()
        for b in range(3):
            k[b, :, t[b]:] = np.nan
            v[b, :, t[b]:] = np.nan
        caches.append((k, v))
    logits, new_kv = oracle.stack_decode(tokens[np.arange(3), t], t, layers, caches, fn, embed, lm, cos, sin, **kw)
    assert np.allclose(logits, full[np.arange(3), t], rtol=0, atol=1e-11)
    assert np.all(np.isfinite(logits))
    # the new token's K of the first layer is the prefill's K at that slot
    _, kf, _ = oracle.decoder_layer(embed[tokens], layers[0], cos, sin, **kw)
    assert np.allclose(new_kv[0][0][:, :, 0], kf[np.arange(3), :, t], rtol=0, atol=1e-12)


def test_synth_recipe_is_deterministic_and_shaped():
    wl = synth.WORKLOADS["tiny_f32_b1_s16"]
    a = synth.layer_weights(wl)
    b = synth.layer_weights(wl)
    assert all(np.array_equal(a[k].data, b[k].data) for k in a)
    assert a["wq"].shape == (64, 64) and a["wk"].shape == (32, 64) and a["w_down"].shape == (64, 176)
    assert np.all(a["attn_norm"].data == 1.0)
    x = synth.activations(wl)
    assert x.shape == (1, 16, 64) and x.dtype == "f32"
