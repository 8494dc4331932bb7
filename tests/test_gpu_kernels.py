"""GPU parity of each step against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import NAN_BF16, TOL, assert_close, bf16_stored, f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_dev):
    from llama_decoder_block_gb300 import build, api as a
    build.build()
    assert a.device_status() == 0
    return a


def _rng(seed):
    return np.random.default_rng(seed)


def test_bounded_wait_gives_up_and_reports(api):
    api.wait_probe(2_000_000)           # 2 ms: the probe waits on an mbarrier nothing arrives at
    assert api.device_status() == -4    # LLAMA_ERR_TIMEOUT
    assert api.device_status() == 0     # read-and-clear
    rec = api.timeout_record()          # the wait that gave up: the probe's one thread
    assert 2_000_000 <= rec["waited_ns"] < 1_000_000_000 and rec["polls"] > 0
    assert rec["thread"] == 0 and rec["block"] == (0, 0) and rec["grid"] == (1, 1)
    x = torch.ones(4, 256, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    api.rmsnorm(x, torch.ones(256, dtype=torch.bfloat16, device="cuda"), y, 1e-5)   # the context still works
    torch.cuda.synchronize()
    assert torch.allclose(y.float(), torch.ones_like(y.float()), atol=1e-2)


@pytest.mark.parametrize("rows,d,dt", [(1, 4096, "bf16"), (37, 4096, "bf16"), (2048, 4096, "bf16"),
                                       (64, 768, "bf16"), (40, 1024, "bf16"), (16, 64, "f32"), (33, 4096, "f32")])
def test_rmsnorm(api, rows, d, dt):
    rng = _rng(rows * 7 + d)
    x = rng.standard_normal((rows, d)) * 3
    g = 1 + 0.1 * rng.standard_normal(d)
    if dt == "bf16":
        xs, gs = bf16_stored(x), bf16_stored(g)
    else:
        from llama_decoder_block_gb300.synth import Stored
        xs, gs = Stored(x.astype(np.float32), "f32"), Stored(g.astype(np.float32), "f32")
    xd, gd = to_dev(xs), to_dev(gs)
    y = torch.empty_like(xd)
    api.rmsnorm(xd, gd, y, 1e-5)
    ref = oracle.rms_norm(xs.f64(), gs.f64(), 1e-5)
    assert_close(f64(y), ref, TOL[dt], "rmsnorm")
    assert api.device_status() == 0


@pytest.mark.parametrize("rows,d,dt", [(1, 4096, "bf16"), (37, 4096, "bf16"), (2048, 4096, "bf16"),
                                       (64, 768, "bf16"), (40, 1024, "bf16"), (9, 100, "bf16"), (16, 64, "f32"),
                                       (33, 4096, "f32")])
def test_layernorm(api, rows, d, dt):
    # rows with a large common offset: the centring must happen before the square
    rng = _rng(rows * 11 + d)
    x = 4.0 + rng.standard_normal((rows, d)) * 2
    g = 1 + 0.1 * rng.standard_normal(d)
    bt = 0.1 * rng.standard_normal(d)
    if dt == "bf16":
        xs, gs, bs = bf16_stored(x), bf16_stored(g), bf16_stored(bt)
    else:
        from llama_decoder_block_gb300.synth import Stored
        xs, gs, bs = (Stored(v.astype(np.float32), "f32") for v in (x, g, bt))
    xd, gd, bd = to_dev(xs), to_dev(gs), to_dev(bs)
    y = torch.empty_like(xd)
    api.layernorm(xd, gd, bd, y, 1e-5)
    ref = oracle.layer_norm(xs.f64(), gs.f64(), bs.f64(), 1e-5)
    assert_close(f64(y), ref, TOL[dt], "layernorm")
    assert api.device_status() == 0


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 520, 200), (1000, 2048, 4096), (64, 6144, 4096)])
@pytest.mark.parametrize("out_f32", [False, True])
def test_linear_bf16(api, M, N, K, out_f32):
    rng = _rng(M + N + K)
    a = bf16_stored(rng.standard_normal((M, K)))
    b = bf16_stored(0.02 * rng.standard_normal((N, K)))
    c = torch.empty(M, N, dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    api.linear_bf16(to_dev(a), to_dev(b), c)
    ref = oracle.linear(a.f64(), b.f64())
    # fp32 output: only fp32 accumulation error; bf16 output: the final rounding too
    assert_close(f64(c), ref, 1e-3 if out_f32 else TOL["bf16"], f"linear {M}x{N}x{K}")
    assert api.device_status() == 0


# Shapes that select each tile form on a 152-SM GB300 (the row blocks pair up when M is a
# multiple of 256): two-SM products on 256-column tiles (M = 256, N = 17448: 69 tiles of 256
# in one round against 78 of 224 in two; the last tile holds 40 columns), B shared by
# multicast on 224-column tiles (M = 256, N = 456: two full tiles and an 8-column one), and
# one CTA per tile (M = 384: three row blocks).
TILE_FORM_SHAPES = [(256, 17448, 256), (256, 456, 256), (384, 456, 256)]


@pytest.mark.parametrize("M,N,K", TILE_FORM_SHAPES)
@pytest.mark.parametrize("out_f32", [False, True])
def test_linear_tile_forms(api, M, N, K, out_f32):
    rng = _rng(M * 3 + N + K)
    a = bf16_stored(rng.standard_normal((M, K)))
    b = bf16_stored(0.02 * rng.standard_normal((N, K)))
    c = torch.empty(M, N, dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    api.linear_bf16(to_dev(a), to_dev(b), c)
    ref = oracle.linear(a.f64(), b.f64())
    assert_close(f64(c), ref, 1e-3 if out_f32 else TOL["bf16"], f"linear {M}x{N}x{K}")
    assert api.device_status() == 0


@pytest.mark.parametrize("M,N,K", [(256, 17408, 256), (256, 384, 256), (384, 384, 256)])
def test_linear_residual_tile_forms(api, M, N, K):
    # the same three forms with N % 128 == 0, as this entry point requires (17408: 68 tiles of
    # 256 in one round against 78 of 224 in two; 384: a 224-column tile and a 160-column one)
    rng = _rng(M * 5 + N + K)
    a = bf16_stored(rng.standard_normal((M, K)))
    b = bf16_stored(0.02 * rng.standard_normal((N, K)))
    r = bf16_stored(rng.standard_normal((M, N)))
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.linear_residual(to_dev(a), to_dev(b), to_dev(r), out)
    ref = r.f64() + oracle.linear(a.f64(), b.f64())
    assert_close(f64(out), ref, TOL["bf16"], f"linear + residual {M}x{N}x{K}")
    assert api.device_status() == 0


@pytest.mark.parametrize("M,I,K", [(256, 384, 256), (256, 9728, 256), (384, 384, 256)])
def test_linear_swiglu_tile_forms(api, M, I, K):
    # M = 256: two-SM products (the even CTA holds the gate rows, the odd one the up rows), in
    # 240-column tiles at I = 384 (4 tiles, the last with 24 of its 120 columns valid) and in
    # 256-column tiles at I = 9728 (76 tiles: one round of pairs, where 240 would take two);
    # M = 384: one CTA per tile
    rng = _rng(M * 7 + I + K)
    x = bf16_stored(rng.standard_normal((M, K)))
    wg = bf16_stored(0.05 * rng.standard_normal((I, K)))
    wu = bf16_stored(0.05 * rng.standard_normal((I, K)))
    a = torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
    api.linear_swiglu(to_dev(x), to_dev(wg), to_dev(wu), a)
    ref = oracle.silu(oracle.linear(x.f64(), wg.f64())) * oracle.linear(x.f64(), wu.f64())
    assert_close(f64(a), ref, TOL["bf16"], f"gate/up + SiLU*up {M}x{I}x{K}")
    assert api.device_status() == 0


def _attn_dims(api, H, G):
    return api.Dims(H * 128, H, G, 128, 128, 1e-5, torch.bfloat16)


def _cache_with_nan_tail(rng, B, G, T_max, valid):
    """[B, G, T_max, 128] bf16 with N(0,1) in slots < valid[b] and NaN beyond (must never be read)."""
    vals = rng.standard_normal((B, G, T_max, 128))
    st = bf16_stored(vals)
    for b in range(B):
        st.data[b, :, valid[b]:, :] = NAN_BF16
    return st


@pytest.mark.parametrize("B,S,H,G", [(2, 300, 4, 2), (1, 128, 2, 2), (1, 520, 8, 1), (2, 256, 8, 2), (1, 1, 4, 4)])
def test_attention_prefill(api, B, S, H, G):
    rng = _rng(B * 1000 + S + H * 10 + G)
    T_max = S + 37
    q = bf16_stored(rng.standard_normal((B, H, S, 128)))
    kc = _cache_with_nan_tail(rng, B, G, T_max, [S] * B)
    vc = _cache_with_nan_tail(rng, B, G, T_max, [S] * B)
    out = torch.empty(B, S, H * 128, dtype=torch.bfloat16, device="cuda")
    api.attention_prefill(_attn_dims(api, H, G), to_dev(q), to_dev(kc), to_dev(vc), out)
    pos = np.tile(np.arange(S), (B, 1))
    ref = oracle.attention(q.f64(), kc.f64()[:, :, :S], vc.f64()[:, :, :S], pos, np.full(B, S))
    gpu = f64(out).reshape(B, S, H, 128).transpose(0, 2, 1, 3)
    assert_close(gpu, ref, TOL["bf16"], "attention prefill")
    assert api.device_status() == 0


def test_attention_prefill_mask_and_group_map_are_exact(api):
    # q = 0: every visible key gets weight 1/(i+1).  V row j of group g is one-hot at column
    # (j + 17 g) % 128, so the nonzero columns of O[b, h, i] name exactly the keys and the group read.
    B, S, H, G = 1, 128, 8, 2
    q = torch.zeros(B, H, S, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(B, G, S, 128, device="cuda").to(torch.bfloat16)
    v = torch.zeros(B, G, S, 128, dtype=torch.bfloat16, device="cuda")
    for g in range(G):
        for j in range(S):
            v[0, g, j, (j + 17 * g) % 128] = 1.0
    out = torch.empty(B, S, H * 128, dtype=torch.bfloat16, device="cuda")
    api.attention_prefill(_attn_dims(api, H, G), q, k, v, out)
    o = f64(out).reshape(S, H, 128)
    for h in range(H):
        g = h // (H // G)
        for i in range(S):
            expect = {(j + 17 * g) % 128 for j in range(i + 1)}
            got = set(np.nonzero(o[i, h])[0].tolist())
            assert got == expect, (h, i)
            assert np.allclose(o[i, h][list(expect)], 1.0 / (i + 1), rtol=1e-2)


@pytest.mark.parametrize("H,G", [(8, 2), (4, 4), (8, 1), (32, 8), (16, 1), (32, 1), (32, 2)])
def test_attention_decode(api, H, G):
    rng = _rng(H * 31 + G)
    positions = np.array([0, 1, 127, 128, 511, 512, 1024, 1099], dtype=np.int32)
    B, T_max = len(positions), 1100
    q = bf16_stored(rng.standard_normal((B, H, 128)))
    kc = _cache_with_nan_tail(rng, B, G, T_max, positions + 1)
    vc = _cache_with_nan_tail(rng, B, G, T_max, positions + 1)
    dims = _attn_dims(api, H, G)
    ws = api.workspace(api.attention_decode_workspace_bytes(dims, B, T_max), "cuda")
    out = torch.empty(B, H * 128, dtype=torch.bfloat16, device="cuda")
    api.attention_decode(dims, to_dev(q), to_dev(kc), to_dev(vc), torch.from_numpy(positions).cuda(), out, ws)
    k64, v64 = kc.f64(), vc.f64()
    for b, p in enumerate(positions):
        ref = oracle.attention(q.f64()[b:b + 1, :, None, :], k64[b:b + 1, :, :p + 1], v64[b:b + 1, :, :p + 1],
                               np.array([[p]]), np.array([p + 1]))[0, :, 0, :]
        assert_close(f64(out)[b].reshape(H, 128), ref, TOL["bf16"], f"decode attention b={b} p={p}")
    assert api.device_status() == 0


@pytest.mark.parametrize("H,G,positions", [(8, 1, [4095, 0, 2000]), (32, 8, [4095, 3, 130, 4000]),
                                           (4, 4, [255, 256, 257])])
def test_attention_decode_long_and_short_sequences(api, H, G, positions):
    # the CTAs split the (sequence, KV head, key tile) axis evenly, so a long sequence next to
    # short ones is cut into many segments that the combine kernel merges
    rng = _rng(H + 7 * G + len(positions))
    positions = np.array(positions, dtype=np.int32)
    B, T_max = len(positions), 4096
    q = bf16_stored(rng.standard_normal((B, H, 128)))
    kc = _cache_with_nan_tail(rng, B, G, T_max, positions + 1)
    vc = _cache_with_nan_tail(rng, B, G, T_max, positions + 1)
    dims = _attn_dims(api, H, G)
    ws = api.workspace(api.attention_decode_workspace_bytes(dims, B, T_max), "cuda")
    out = torch.empty(B, H * 128, dtype=torch.bfloat16, device="cuda")
    api.attention_decode(dims, to_dev(q), to_dev(kc), to_dev(vc), torch.from_numpy(positions).cuda(), out, ws)
    k64, v64 = kc.f64(), vc.f64()
    for b, p in enumerate(positions):
        ref = oracle.attention(q.f64()[b:b + 1, :, None, :], k64[b:b + 1, :, :p + 1], v64[b:b + 1, :, :p + 1],
                               np.array([[p]]), np.array([p + 1]))[0, :, 0, :]
        assert_close(f64(out)[b].reshape(H, 128), ref, TOL["bf16"], f"decode attention b={b} p={p}")
    assert api.device_status() == 0


def test_attention_decode_more_sequences_than_one_launch_holds(api):
    # 1030 sequences: the library runs them as launches of at most 1024 sequences
    B, H, G, T_max = 1030, 8, 2, 200
    rng = _rng(1030)
    positions = rng.integers(0, T_max, size=B).astype(np.int32)
    positions[[0, 1023, 1024, 1029]] = [T_max - 1, 0, T_max - 1, 5]
    q = torch.from_numpy(rng.standard_normal((B, H, 128)).astype(np.float32)).to(torch.bfloat16).cuda()
    kc = torch.from_numpy(rng.standard_normal((B, G, T_max, 128)).astype(np.float32)).to(torch.bfloat16).cuda()
    vc = torch.from_numpy(rng.standard_normal((B, G, T_max, 128)).astype(np.float32)).to(torch.bfloat16).cuda()
    dims = _attn_dims(api, H, G)
    ws = api.workspace(api.attention_decode_workspace_bytes(dims, B, T_max), "cuda")
    out = torch.empty(B, H * 128, dtype=torch.bfloat16, device="cuda")
    api.attention_decode(dims, q, kc, vc, torch.from_numpy(positions).cuda(), out, ws)
    assert api.device_status() == 0
    o = f64(out).reshape(B, H, 128)
    for b in [0, 1, 511, 1022, 1023, 1024, 1025, 1029] + rng.integers(0, B, size=12).tolist():
        p = int(positions[b])
        ref = oracle.attention(f64(q[b:b + 1])[:, :, None, :], f64(kc[b:b + 1, :, :p + 1]),
                               f64(vc[b:b + 1, :, :p + 1]), np.array([[p]]), np.array([p + 1]))[0, :, 0, :]
        assert_close(o[b], ref, TOL["bf16"], f"decode attention b={b} p={p}")


def test_attention_decode_reports_out_of_range_positions(api):
    B, H, G, T_max = 3, 4, 2, 256
    dims = _attn_dims(api, H, G)
    q = torch.randn(B, H, 128, device="cuda").to(torch.bfloat16)
    kc = torch.randn(B, G, T_max, 128, device="cuda").to(torch.bfloat16)
    vc = torch.randn(B, G, T_max, 128, device="cuda").to(torch.bfloat16)
    ws = api.workspace(api.attention_decode_workspace_bytes(dims, B, T_max), "cuda")
    out = torch.empty(B, H * 128, dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([5, T_max, 7], dtype=torch.int32, device="cuda")
    api.attention_decode(dims, q, kc, vc, pos, out, ws)
    assert api.device_status() == -5
    assert torch.all(out[1] == 0) and torch.all(torch.isfinite(out.float()))


def _one_ulp(gpu, ref, what):
    """A bf16 result of one fp32-accumulated step: within one bf16 ulp (2^-8 relative) plus the
    accumulation error, which 1e-3 of the row's rms bounds generously."""
    scale = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bad = np.abs(gpu - ref) > 2.0 ** -8 * np.abs(ref) + 1e-3 * scale
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond one bf16 ulp, first at {np.argwhere(bad)[0]}"


def _norm_inputs(rng, M, K, scale=3.0):
    x = bf16_stored(scale * rng.standard_normal((M, K)))
    g = bf16_stored(1 + 0.1 * rng.standard_normal(K))
    return x, g


def _check_prologue(api, xd, gd, xn, eps, what):
    """The GEMM prologue's normalised rows are bit for bit those of the standalone RMSNorm (same
    arithmetic, same order), and within one rounding of the oracle's."""
    y = torch.empty_like(xd)
    api.rmsnorm(xd, gd, y, eps)
    assert torch.equal(xn.view(-1), y.view(-1)), f"{what}: prologue rows differ from llama_rmsnorm"


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 520, 256), (1000, 2048, 4096), (7, 32000, 4096),
                                   (2048, 8192, 4096), (130, 264, 200)])
@pytest.mark.parametrize("out_f32", [False, True])
def test_norm_linear_fused(api, M, N, K, out_f32):
    # RMSNorm in the GEMM's prologue: the GEMM normalises the rows into xn and multiplies xn, so
    # the result is the oracle's RMSNorm (rounded where it stores its output) followed by the
    # product.  (2048 x 8192 x 4096: several tiles per CTA; K = 64, 200: the generic prologue.)
    rng = _rng(M * 3 + N + K)
    x, g = _norm_inputs(rng, M, K)
    w = bf16_stored(0.02 * rng.standard_normal((N, K)))
    c = torch.empty(M, N, dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    xd, gd = to_dev(x), to_dev(g)
    xn = api.norm_linear_bf16(xd, gd, 1e-5, to_dev(w), c)
    assert api.device_status() == 0
    xn_ref = oracle.round_bf16(oracle.rms_norm(x.f64(), g.f64(), 1e-5))
    assert_close(f64(xn), xn_ref, TOL["bf16"], f"norm prologue {M}x{K}")
    ref = oracle.linear(xn_ref, w.f64())
    assert_close(f64(c), ref, TOL["bf16"], f"norm + linear {M}x{N}x{K}")
    # the product of the rows the prologue wrote: fp32 output within accumulation error, bf16
    # output within one ulp (the oracle's fp64 row rounds to the other bf16 neighbour at ~1e-4 of
    # the elements, which moves an output by up to a few 1e-3)
    exact = oracle.linear(f64(xn), w.f64())
    if out_f32:
        assert_close(f64(c), exact, 1e-4, f"norm + linear {M}x{N}x{K}, fp32 out, on the prologue's rows")
    else:
        _one_ulp(f64(c), exact, f"norm + linear {M}x{N}x{K}")
    if K % 256 == 0:
        _check_prologue(api, xd, gd, xn, 1e-5, f"norm + linear {M}x{N}x{K}")


@pytest.mark.parametrize("M,I,K", [(130, 384, 256), (1000, 11008, 4096), (64, 1024, 4096), (2048, 11008, 4096)])
def test_norm_linear_swiglu_fused(api, M, I, K):
    rng = _rng(M + I + K)
    x, g = _norm_inputs(rng, M, K)
    wg = bf16_stored(0.02 * rng.standard_normal((I, K)))
    wu = bf16_stored(0.02 * rng.standard_normal((I, K)))
    a = torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
    xd, gd = to_dev(x), to_dev(g)
    xn = api.norm_linear_swiglu(xd, gd, 1e-6, to_dev(wg), to_dev(wu), a)
    assert api.device_status() == 0
    xn_ref = oracle.round_bf16(oracle.rms_norm(x.f64(), g.f64(), 1e-6))
    ref = oracle.silu(oracle.linear(xn_ref, wg.f64())) * oracle.linear(xn_ref, wu.f64())
    assert_close(f64(a), ref, TOL["bf16"], f"norm + gate/up {M}x{I}x{K}")
    xg = f64(xn)
    _one_ulp(f64(a), oracle.silu(oracle.linear(xg, wg.f64())) * oracle.linear(xg, wu.f64()),
             f"norm + gate/up {M}x{I}x{K}")
    _check_prologue(api, xd, gd, xn, 1e-6, f"norm + gate/up {M}x{I}x{K}")


@pytest.mark.parametrize("d,H,G,B,S,rope", [(256, 4, 2, 2, 130, "even_odd"), (512, 8, 1, 1, 300, "even_odd"),
                                            (256, 4, 2, 2, 150, "half"), (4096, 32, 8, 1, 256, "even_odd"),
                                            (4096, 32, 8, 3, 700, "even_odd")])
def test_norm_qkv_rope_fused(api, d, H, G, B, S, rope):
    rng = _rng(d + H * 7 + G + B * 13 + S)
    D, T_max = 128, S + 9
    x, g = _norm_inputs(rng, B * S, d, scale=1.0)
    wq = bf16_stored(0.02 * rng.standard_normal((H * D, d)))
    wk = bf16_stored(0.02 * rng.standard_normal((G * D, d)))
    wv = bf16_stored(0.02 * rng.standard_normal((G * D, d)))
    c64, s64 = oracle.rope_tables(1e4, D, T_max)
    c32, s32 = c64.astype(np.float32), s64.astype(np.float32)
    cos, sin = torch.from_numpy(c32).cuda(), torch.from_numpy(s32).cuda()
    kc = torch.full((B, G, T_max, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    q = torch.empty(B, H, S, D, dtype=torch.bfloat16, device="cuda")
    dims = api.Dims(d, H, G, D, 128, 1e-5, torch.bfloat16, 1 if rope == "half" else 0)
    xd, gd = to_dev(x), to_dev(g)
    xn = api.norm_qkv_rope(dims, xd.view(B, S, d), gd, to_dev(wq), to_dev(wk), to_dev(wv), cos, sin, kc, vc, q)
    assert api.device_status() == 0
    xn_ref = oracle.round_bf16(oracle.rms_norm(x.f64(), g.f64(), 1e-5)).reshape(B, S, d)
    rot = oracle.layer.ROPE_STYLES[rope]
    cc, ss = c32.astype(np.float64)[:S][None, None], s32.astype(np.float64)[:S][None, None]
    q_ref = rot(oracle.linear(xn_ref, wq.f64()).reshape(B, S, H, D).transpose(0, 2, 1, 3), cc, ss)
    k_ref = rot(oracle.linear(xn_ref, wk.f64()).reshape(B, S, G, D).transpose(0, 2, 1, 3), cc, ss)
    v_ref = oracle.linear(xn_ref, wv.f64()).reshape(B, S, G, D).transpose(0, 2, 1, 3)
    assert_close(f64(q), q_ref, TOL["bf16"], "norm + qkv: q")
    assert_close(f64(kc)[:, :, :S], k_ref, TOL["bf16"], "norm + qkv: k in the cache")
    assert_close(f64(vc)[:, :, :S], v_ref, TOL["bf16"], "norm + qkv: v in the cache")
    assert torch.isnan(kc[:, :, S:].float()).all() and torch.isnan(vc[:, :, S:].float()).all()
    xg = f64(xn).reshape(B, S, d)
    _one_ulp(f64(q), rot(oracle.linear(xg, wq.f64()).reshape(B, S, H, D).transpose(0, 2, 1, 3), cc, ss),
             "norm + qkv: q")
    _check_prologue(api, xd, gd, xn, 1e-5, "norm + qkv")
