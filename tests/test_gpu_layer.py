"""GPU parity of the whole layer (prefill, decode) and of the stack against the fp64 oracle."""
import os

import numpy as np
import gpu_util
import pytest
import torch

import oracle
from gpu_util import (NAN_BF16, TOL, assert_close, assert_close_layer_full, bf16_stored, dims_of, f64, oracle_kw,
                      tables, to_dev)
from llama_decoder_block_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_dev):
    from llama_decoder_block_gb300 import build, api as a
    build.build()
    assert a.device_status() == 0
    return a


def _weights(wl, layer=0):
    st = synth.layer_weights(wl, layer)
    return st, {k: to_dev(v) for k, v in st.items()}


def _run_prefill(api, wl, extra_T=5, max_pos=None):
    L = wl.layer
    B, S = wl.B, wl.S
    T_max = S + extra_T
    max_pos = max_pos or T_max
    st, w = _weights(wl)
    xs = synth.activations(wl)
    x = to_dev(xs)
    out = torch.empty_like(x)
    cos, sin, c64, s64 = tables(L, max_pos, oracle)
    dt = x.dtype
    kc = torch.full((B, L.n_kv_heads, T_max, L.head_dim), float("nan"), dtype=dt, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    dims = dims_of(L)
    ws = api.workspace(api.prefill_workspace_bytes(dims, B, S), "cuda")
    api.layer_prefill(dims, w, x, out, cos, sin, kc, vc, ws)
    assert api.device_status() == 0
    return st, xs, c64, s64, out, kc, vc


def _check_prefill(api, wl, prefix=None, full_width=False):
    L = wl.layer
    st, xs, c64, s64, out, kc, vc = _run_prefill(api, wl)
    x64 = xs.f64()
    S_ref = prefix or wl.S
    w64 = {k: v.f64() for k, v in st.items()}
    ref, k_ref, v_ref = oracle.decoder_layer(x64[:, :S_ref], w64, c64, s64, store_bf16=(L.dtype == "bf16"),
                                             **oracle_kw(L))
    tol = TOL[L.dtype]
    if full_width:
        print(assert_close_layer_full(f64(out)[:, :S_ref], ref, f"{wl.name} out"))
    else:
        assert_close(f64(out)[:, :S_ref], ref, tol, f"{wl.name} out")
    assert_close(f64(kc)[:, :, :S_ref], k_ref, tol, f"{wl.name} cache K")
    assert_close(f64(vc)[:, :, :S_ref], v_ref, tol, f"{wl.name} cache V")
    # slots >= S are never written
    assert torch.isnan(kc[:, :, wl.S:].float()).all() and torch.isnan(vc[:, :, wl.S:].float()).all()


def test_prefill_tiny_fp32_config(api):
    _check_prefill(api, synth.WORKLOADS["tiny_f32_b1_s16"])


@pytest.mark.parametrize("H,G,B,S", [(4, 2, 2, 200), (2, 2, 1, 128), (8, 1, 1, 300), (4, 4, 3, 65), (16, 1, 1, 140),
                                     (32, 2, 1, 70), (4, 2, 3, 1), (4, 2, 1, 129)])
def test_prefill_bf16_small(api, H, G, B, S):
    base = synth.WORKLOADS["gqa8b_bf16_b4_s4096"]
    wl = synth.scaled(base, d_model=256, n_heads=H, n_kv_heads=G, d_inter=384, B=B, S=S,
                      name=f"bf16_d256_h{H}_g{G}_b{B}_s{S}")
    _check_prefill(api, wl)


@pytest.mark.parametrize("H,G", [(4, 2), (16, 1)])
def test_prefill_bf16_half_split_rope(api, H, G):
    base = synth.WORKLOADS["gqa8b_bf16_b4_s4096"]
    wl = synth.scaled(base, d_model=256, n_heads=H, n_kv_heads=G, d_inter=384, B=2, S=150, rope_style="half",
                      name=f"bf16_half_rope_h{H}_g{G}")
    _check_prefill(api, wl)


def test_prefill_fp32_half_split_rope(api):
    base = synth.WORKLOADS["tiny_f32_b1_s16"]
    wl = synth.scaled(base, d_model=96, n_heads=6, n_kv_heads=3, head_dim=16, d_inter=160, B=2, S=37,
                      rope_style="half", name="f32_half_rope")
    _check_prefill(api, wl)


def test_prefill_fp32_gqa_ragged(api):
    base = synth.WORKLOADS["tiny_f32_b1_s16"]
    wl = synth.scaled(base, d_model=96, n_heads=6, n_kv_heads=3, head_dim=16, d_inter=160, B=2, S=37,
                      name="f32_d96_h6_g3_b2_s37")
    _check_prefill(api, wl)


def test_prefill_mha7b_full_size(api):
    _check_prefill(api, synth.WORKLOADS["mha7b_bf16_b1_s2048"], full_width=True)


def test_prefill_gqa8b_full_size_causal_prefix(api):
    # the GPU runs B=4, S=4096; rows < 256 depend only on tokens < 256 (causality), so the
    # oracle's 256-token run is their exact reference
    _check_prefill(api, synth.WORKLOADS["gqa8b_bf16_b4_s4096"], prefix=256, full_width=True)


def _cache_with_history(wl, T_max, start, seed):
    """[B, G, T_max, D] K and V caches: N(0,1) in slots < start[b] (the history), NaN elsewhere."""
    L = wl.layer
    rng = np.random.default_rng(seed)
    shape = (wl.B, L.n_kv_heads, T_max, L.head_dim)
    out = []
    for _ in range(2):
        vals = rng.standard_normal(shape)
        st = bf16_stored(vals) if L.dtype == "bf16" else synth.Stored(vals.astype(np.float32), "f32")
        for b in range(wl.B):
            st.data[b, :, start[b]:] = NAN_BF16 if L.dtype == "bf16" else np.nan
        out.append(st)
    return out


def _check_chunk(api, wl, start, lengths, T_max, full_width=False):
    L = wl.layer
    B, S = wl.B, wl.S
    start = np.asarray(start, dtype=np.int32)
    lens = np.full(B, S, dtype=np.int32) if lengths is None else np.asarray(lengths, dtype=np.int32)
    st, w = _weights(wl)
    xs = synth.activations(wl)
    x = to_dev(xs)
    out = torch.empty_like(x)
    ks, vs = _cache_with_history(wl, T_max, start, wl.seed + 7)
    kc, vc = to_dev(ks), to_dev(vs)
    cos, sin, c64, s64 = tables(L, T_max, oracle)
    dims = dims_of(L)
    ws = api.workspace(api.prefill_workspace_bytes(dims, B, S), "cuda")
    api.layer_prefill_chunk(dims, w, x, out, cos, sin, torch.from_numpy(start).cuda(), kc, vc, ws,
                            lengths=None if lengths is None else torch.from_numpy(lens).cuda())
    assert api.device_status() == 0
    w64 = {k: v.f64() for k, v in st.items()}
    x64, k64, v64 = xs.f64(), ks.f64(), vs.f64()
    out_h, kc_h, vc_h = f64(out), f64(kc), f64(vc)
    tol = TOL[L.dtype]
    for b in range(B):
        p0, n = int(start[b]), int(lens[b])
        ref, k_new, v_new = oracle.decoder_layer(x64[b:b + 1, :n], w64, c64, s64, past_k=k64[b:b + 1],
                                                 past_v=v64[b:b + 1], past_len=np.array([p0]),
                                                 store_bf16=(L.dtype == "bf16"), **oracle_kw(L))
        if full_width:
            print(assert_close_layer_full(out_h[b, :n], ref[0], f"chunk out b={b} start={p0} len={n}"))
        else:
            assert_close(out_h[b, :n], ref[0], tol, f"chunk out b={b} start={p0} len={n}")
        assert_close(kc_h[b, :, p0:p0 + n], k_new[0], tol, f"chunk cache K b={b}")
        assert_close(vc_h[b, :, p0:p0 + n], v_new[0], tol, f"chunk cache V b={b}")
        others = np.ones(T_max, bool)
        others[p0:p0 + n] = False
        assert np.array_equal(kc_h[b][:, others], k64[b][:, others], equal_nan=True)
        assert np.array_equal(vc_h[b][:, others], v64[b][:, others], equal_nan=True)


@pytest.mark.parametrize("H,G,start,lengths,S,T_max", [
    (4, 2, [0, 37, 300], [150, 90, 1], 150, 512),      # ragged, one from position 0
    (8, 1, [130, 5], None, 200, 400),                   # MQA-sized groups, tile-unaligned starts
    (4, 4, [1000], None, 300, 1400),                    # long history: many key tiles, two masked
    (2, 2, [256, 128], [128, 100], 128, 400),           # tile-aligned starts
])
def test_prefill_chunk_bf16(api, H, G, start, lengths, S, T_max):
    base = synth.WORKLOADS["gqa8b_bf16_b4_s4096"]
    wl = synth.scaled(base, d_model=256, n_heads=H, n_kv_heads=G, d_inter=384, B=len(start), S=S,
                      name=f"chunk_bf16_h{H}_g{G}_s{S}")
    _check_chunk(api, wl, start, lengths, T_max)


def test_prefill_chunk_gqa8b_full_width(api):
    # the GQA-8B layer at full width on top of long cached histories (ragged chunk)
    base = synth.WORKLOADS["gqa8b_bf16_b4_s4096"]
    wl = synth.scaled(base, B=2, S=256, name="chunk_gqa8b_full_width")
    _check_chunk(api, wl, [1000, 3700], [256, 200], 4096, full_width=True)


def test_prefill_chunk_fp32(api):
    base = synth.WORKLOADS["tiny_f32_b1_s16"]
    wl = synth.scaled(base, B=2, S=9, name="chunk_f32_tiny")
    _check_chunk(api, wl, [0, 20], [9, 4], 40)


def test_two_chunks_equal_one_prefill(api):
    # prefill(prompt[:100]) then the chunk prompt[100:] on top of it: the same outputs and cache
    # as prefill(prompt) in one call
    base = synth.WORKLOADS["gqa8b_bf16_b4_s4096"]
    wl = synth.scaled(base, d_model=256, n_heads=4, n_kv_heads=2, d_inter=384, B=2, S=256, name="two_chunks")
    L = wl.layer
    st, w = _weights(wl)
    x = to_dev(synth.activations(wl))
    T_max = 300
    cos, sin, _, _ = tables(L, T_max, oracle)
    dims = dims_of(L)
    ws = api.workspace(api.prefill_workspace_bytes(dims, wl.B, wl.S), "cuda")
    shape = (wl.B, L.n_kv_heads, T_max, L.head_dim)
    k1, v1 = torch.zeros(shape, dtype=torch.bfloat16, device="cuda"), torch.zeros(shape, dtype=torch.bfloat16,
                                                                                 device="cuda")
    k2, v2 = k1.clone(), v1.clone()
    full = torch.empty_like(x)
    api.layer_prefill(dims, w, x, full, cos, sin, k1, v1, ws)
    a = torch.empty(wl.B, 100, L.d_model, dtype=torch.bfloat16, device="cuda")
    c = torch.empty(wl.B, 156, L.d_model, dtype=torch.bfloat16, device="cuda")
    zeros = torch.zeros(wl.B, dtype=torch.int32, device="cuda")
    api.layer_prefill_chunk(dims, w, x[:, :100].contiguous(), a, cos, sin, zeros, k2, v2, ws)
    api.layer_prefill_chunk(dims, w, x[:, 100:].contiguous(), c, cos, sin, zeros + 100, k2, v2, ws)
    assert api.device_status() == 0
    assert_close(f64(torch.cat([a, c], dim=1)), f64(full), TOL["bf16"], "chunked vs whole prefill")
    assert_close(f64(k2), f64(k1), TOL["bf16"], "chunked vs whole cache K")
    assert_close(f64(v2), f64(v1), TOL["bf16"], "chunked vs whole cache V")


def test_prefill_chunk_out_of_range_is_reported(api):
    base = synth.WORKLOADS["gqa8b_bf16_b4_s4096"]
    wl = synth.scaled(base, d_model=256, n_heads=4, n_kv_heads=2, d_inter=384, B=2, S=64, name="chunk_bounds")
    L = wl.layer
    _, w = _weights(wl)
    x = to_dev(synth.activations(wl))
    out = torch.empty_like(x)
    T_max = 100
    cos, sin, _, _ = tables(L, T_max, oracle)
    dims = dims_of(L)
    ws = api.workspace(api.prefill_workspace_bytes(dims, wl.B, wl.S), "cuda")
    kc = torch.zeros(wl.B, L.n_kv_heads, T_max, L.head_dim, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    start = torch.tensor([10, 50], dtype=torch.int32, device="cuda")   # 50 + 64 > 100
    api.layer_prefill_chunk(dims, w, x, out, cos, sin, start, kc, vc, ws)
    assert api.device_status() == -5
    assert torch.all(kc[1] == 0) and torch.all(vc[1] == 0)             # the bad sequence wrote nothing
    assert torch.isfinite(out[0].float()).all()


def _run_decode(api, wl, positions=None, nan_beyond=True, sample=None, full_width=False):
    L = wl.layer
    st, w = _weights(wl)
    pos, ks, vs = synth.decode_state(wl)
    if positions is not None:
        pos = np.asarray(positions, dtype=np.int32)
    if nan_beyond:
        for b in range(wl.B):
            ks.data[b, :, pos[b] + 1:] = NAN_BF16 if L.dtype == "bf16" else np.nan
            vs.data[b, :, pos[b] + 1:] = NAN_BF16 if L.dtype == "bf16" else np.nan
    xs = synth.activations(wl)
    x = to_dev(xs)
    out = torch.empty_like(x)
    kc, vc = to_dev(ks), to_dev(vs)
    cos, sin, c64, s64 = tables(L, wl.T_max, oracle)
    dims = dims_of(L)
    ws = api.workspace(api.decode_workspace_bytes(dims, wl.B, wl.T_max), "cuda")
    api.layer_decode(dims, w, x, out, cos, sin, torch.from_numpy(pos).cuda(), kc, vc, ws)
    assert api.device_status() == 0
    w64 = {k: v.f64() for k, v in st.items()}
    tol = TOL[L.dtype]
    x64 = xs.f64()
    out_h = f64(out)
    for b in (range(wl.B) if sample is None else sample):
        p = int(pos[b])
        ks64 = synth.Stored(ks.data[b:b + 1], ks.dtype).f64()
        vs64 = synth.Stored(vs.data[b:b + 1], vs.dtype).f64()
        ref, k_new, v_new = oracle.decoder_layer(
            x64[b:b + 1, None, :], w64, c64, s64, past_k=ks64, past_v=vs64,
            past_len=np.array([p]), store_bf16=(L.dtype == "bf16"), **oracle_kw(L))
        kc_h, vc_h = f64(kc[b]), f64(vc[b])
        if full_width:
            assert_close_layer_full(out_h[b], ref[0, 0], f"decode out b={b} p={p}")
        else:
            assert_close(out_h[b], ref[0, 0], tol, f"decode out b={b} p={p}")
        assert_close(kc_h[:, p], k_new[0, :, 0], tol, f"decode cache K slot b={b} p={p}")
        assert_close(vc_h[:, p], v_new[0, :, 0], tol, f"decode cache V slot b={b} p={p}")
        # every other slot is untouched (bitwise, NaN included)
        others = np.ones(wl.T_max, bool)
        others[p] = False
        assert np.array_equal(kc_h[:, others], ks64[0][:, others], equal_nan=True)
        assert np.array_equal(vc_h[:, others], vs64[0][:, others], equal_nan=True)


def test_decode_bf16_small_edge_positions(api):
    base = synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"]
    wl = synth.scaled(base, d_model=256, n_heads=8, n_kv_heads=2, d_inter=384, B=6, T_max=600,
                      name="decode_bf16_d256_b6_t600")
    _run_decode(api, wl, positions=[0, 1, 300, 511, 512, 599])


@pytest.mark.parametrize("H,G,rope", [(16, 1, "even_odd"), (8, 2, "half"), (32, 1, "half")])
def test_decode_bf16_mqa_and_half_split_rope(api, H, G, rope):
    base = synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"]
    wl = synth.scaled(base, d_model=256, n_heads=H, n_kv_heads=G, d_inter=384, B=5, T_max=700, rope_style=rope,
                      name=f"decode_bf16_h{H}_g{G}_{rope}")
    _run_decode(api, wl, positions=[0, 130, 511, 650, 699])


@pytest.mark.parametrize("B", [1, 70])
def test_decode_bf16_token_tiles(api, B):
    # the weight-streaming GEMMs take the tokens as the N = 64 operand: one token, and two token
    # tiles with a ragged second one (70 = 64 + 6); positions over the whole cache, 0 included
    base = synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"]
    wl = synth.scaled(base, d_model=256, n_heads=8, n_kv_heads=2, d_inter=384, B=B, T_max=300, pos_lo=0, pos_hi=300,
                      name=f"decode_bf16_b{B}_t300")
    _run_decode(api, wl, positions=[0] if B == 1 else None)


def test_decode_fp32_half_split_rope(api):
    base = synth.WORKLOADS["tiny_f32_b1_s16"]
    wl = synth.scaled(base, kind="decode", B=4, S=0, T_max=40, pos_lo=0, pos_hi=40, rope_style="half",
                      name="decode_f32_half_rope")
    _run_decode(api, wl)


def test_decode_fp32_small(api):
    base = synth.WORKLOADS["tiny_f32_b1_s16"]
    wl = synth.scaled(base, kind="decode", B=4, S=0, T_max=40, pos_lo=0, pos_hi=40, name="decode_f32_tiny_b4")
    _run_decode(api, wl, positions=[0, 5, 17, 39])


def test_decode_gqa8b_full_size_sampled(api):
    wl = synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"]
    pos = synth.decode_state(wl)[0]
    order = np.argsort(pos)
    _run_decode(api, wl, nan_beyond=False, sample=sorted({int(order[0]), int(order[-1]), 0, 17, 40, 63}),
                full_width=True)


def test_decode_matches_prefill_row(api):
    # "第 10 章：现代 LLaMA 架构" §7: decode of token t over the cache of tokens < t equals
    # row t of the full prefill (here both on the GPU, at the scaled bf16 shape).
    base = synth.WORKLOADS["gqa8b_bf16_b4_s4096"]
    wl = synth.scaled(base, d_model=256, n_heads=4, n_kv_heads=2, d_inter=384, B=2, S=150, name="bf16_pd_b2_s150")
    st, xs, c64, s64, out, kc, vc = _run_prefill(api, wl, extra_T=0)
    L = wl.layer
    _, w = _weights(wl)
    t = wl.S - 1
    x_t = to_dev(xs)[:, t].contiguous()
    y = torch.empty_like(x_t)
    kc2, vc2 = kc.clone(), vc.clone()
    kc2[:, :, t:] = float("nan")
    vc2[:, :, t:] = float("nan")
    dims = dims_of(L)
    cos, sin, _, _ = tables(L, wl.S, oracle)
    ws = api.workspace(api.decode_workspace_bytes(dims, wl.B, wl.S), "cuda")
    api.layer_decode(dims, w, x_t, y, cos, sin, torch.full((wl.B,), t, dtype=torch.int32, device="cuda"), kc2, vc2, ws)
    assert api.device_status() == 0
    assert_close(f64(y), f64(out)[:, t], TOL["bf16"], "decode vs prefill row")


def test_decode_out_of_range_position_is_reported(api):
    base = synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"]
    wl = synth.scaled(base, d_model=256, n_heads=8, n_kv_heads=2, d_inter=384, B=3, T_max=64, name="decode_oob")
    L = wl.layer
    _, w = _weights(wl)
    x = torch.randn(3, 256, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(x)
    kc = torch.randn(3, 2, 64, 128, device="cuda").to(torch.bfloat16)
    vc = torch.randn_like(kc)
    k0, v0 = kc.clone(), vc.clone()
    cos, sin, _, _ = tables(L, 64, oracle)
    dims = dims_of(L)
    ws = api.workspace(api.decode_workspace_bytes(dims, 3, 64), "cuda")
    api.layer_decode(dims, w, x, out, cos, sin, torch.tensor([3, 64, -1], dtype=torch.int32, device="cuda"), kc, vc, ws)
    assert api.device_status() == -5
    assert torch.equal(kc[1:], k0[1:]) and torch.equal(vc[1:], v0[1:])   # bad sequences leave the cache alone


def _stack_case(api, wl, n_layers, prefix=None):
    L = wl.layer
    layers_st = [synth.layer_weights(wl, l) for l in range(n_layers)]
    glob = synth.stack_globals(wl)
    dev_layers = [{k: to_dev(v) for k, v in st.items()} for st in layers_st]
    fn, emb, lm = to_dev(glob["final_norm"]), to_dev(glob["embed"]), to_dev(glob["lm_head"])
    st = api.StackArgs(dims_of(L), dev_layers, fn, emb, lm)
    tokens = torch.from_numpy(glob["tokens"]).cuda()
    logits = torch.empty(wl.B, wl.S, wl.vocab, dtype=torch.float32, device="cuda")
    cos, sin, c64, s64 = tables(L, wl.S, oracle)
    ws = api.workspace(st.workspace_bytes(wl.B, wl.S), "cuda")
    api.stack_forward(st, tokens, logits, cos, sin, ws)
    assert api.device_status() == 0
    S_ref = prefix or wl.S
    ref = oracle.stack_forward(glob["tokens"][:, :S_ref], ({k: v.f64() for k, v in s.items()} for s in layers_st),
                               glob["final_norm"].f64(), glob["embed"].f64(), glob["lm_head"].f64(), c64, s64,
                               store_bf16=(L.dtype == "bf16"), **oracle_kw(L))
    assert_close(f64(logits)[:, :S_ref], ref, TOL[L.dtype], f"{wl.name} logits")


def test_stack_bf16_small(api):
    base = synth.WORKLOADS["stack32_gqa8b_bf16_s8192_v32000"]
    wl = synth.scaled(base, d_model=256, n_heads=4, n_kv_heads=2, d_inter=384, S=130, vocab=1000, n_layers=3,
                      name="stack3_bf16_d256_s130_v1000")
    _stack_case(api, wl, 3)


def test_stack_fp32_tiny(api):
    base = synth.WORKLOADS["tiny_f32_b1_s16"]
    wl = synth.scaled(base, kind="stack", B=2, S=16, vocab=96, n_layers=2, name="stack2_f32_tiny")
    _stack_case(api, wl, 2)


def _stack_decode_setup(api, wl, positions):
    """Device stack, per-layer caches (NaN past each position) and the oracle's inputs."""
    L = wl.layer
    layers_st = [synth.layer_weights(wl, l) for l in range(wl.n_layers)]
    glob = synth.stack_globals(wl)
    nan = NAN_BF16 if L.dtype == "bf16" else np.nan
    pos = np.asarray(positions, dtype=np.int32)
    caches_st = []
    for l in range(wl.n_layers):
        _, ks, vs = synth.decode_state(wl, l)
        for b in range(wl.B):
            ks.data[b, :, pos[b]:] = nan
            vs.data[b, :, pos[b]:] = nan
        caches_st.append((ks, vs))
    dev_layers = [{k: to_dev(v) for k, v in st.items()} for st in layers_st]
    st = api.StackArgs(dims_of(L), dev_layers, to_dev(glob["final_norm"]), to_dev(glob["embed"]),
                       to_dev(glob["lm_head"]))
    caches = [(to_dev(k), to_dev(v)) for k, v in caches_st]
    tokens = glob["tokens"][:, 0].copy()
    return st, caches, caches_st, layers_st, glob, tokens, pos


def _stack_decode_reference(wl, layers_st, caches_st, glob, tokens, pos):
    L = wl.layer
    _, _, c64, s64 = tables(L, wl.T_max, oracle, device="cpu")
    return oracle.stack_decode(tokens, pos, [{k: v.f64() for k, v in s.items()} for s in layers_st],
                               [(k.f64(), v.f64()) for k, v in caches_st], glob["final_norm"].f64(),
                               glob["embed"].f64(), glob["lm_head"].f64(), c64, s64,
                               store_bf16=(L.dtype == "bf16"), **oracle_kw(L))


@pytest.mark.parametrize("vocab,rope", [(512, "even_odd"), (520, "half")])
def test_stack_decode_bf16_small(api, vocab, rope):
    # vocab 512: the LM head streams its weights (split-K); 520: the tiled GEMM
    base = synth.WORKLOADS["stack32_gqa8b_bf16_s8192_v32000"]
    wl = synth.scaled(base, kind="decode", d_model=256, n_heads=4, n_kv_heads=2, d_inter=384, B=5, S=1,
                      T_max=300, pos_lo=0, pos_hi=300, vocab=vocab, n_layers=3, gamma="noisy", rope_style=rope,
                      name=f"stack3_decode_bf16_v{vocab}_{rope}")
    st, caches, caches_st, layers_st, glob, tokens, pos = _stack_decode_setup(api, wl, [0, 1, 150, 257, 299])
    L = wl.layer
    cos, sin, _, _ = tables(L, wl.T_max, oracle)
    logits = torch.empty(wl.B, wl.vocab, dtype=torch.float32, device="cuda")
    ws = api.workspace(api.stack_decode_workspace_bytes(st, wl.B), "cuda")
    api.stack_decode(st, torch.from_numpy(tokens).cuda(), torch.from_numpy(pos).cuda(), logits, cos, sin, caches, ws)
    assert api.device_status() == 0
    ref, new_kv = _stack_decode_reference(wl, layers_st, caches_st, glob, tokens, pos)
    assert_close(f64(logits), ref, TOL["bf16"], "stack decode logits")
    for l, ((kc, vc), (kn, vn)) in enumerate(zip(caches, new_kv)):
        for b, p in enumerate(pos):
            assert_close(f64(kc[b, :, p]), kn[b, :, 0], TOL["bf16"], f"layer {l} K slot b={b}")
            assert_close(f64(vc[b, :, p]), vn[b, :, 0], TOL["bf16"], f"layer {l} V slot b={b}")
            # slots past the new one stay untouched (NaN)
            assert torch.isnan(kc[b, :, p + 1:].float()).all() and torch.isnan(vc[b, :, p + 1:].float()).all()


def test_stack_decode_fp32_tiny(api):
    base = synth.WORKLOADS["tiny_f32_b1_s16"]
    wl = synth.scaled(base, kind="decode", B=3, S=1, T_max=24, pos_lo=0, pos_hi=24, vocab=96, n_layers=2,
                      name="stack2_decode_f32")
    st, caches, caches_st, layers_st, glob, tokens, pos = _stack_decode_setup(api, wl, [0, 9, 23])
    cos, sin, _, _ = tables(wl.layer, wl.T_max, oracle)
    logits = torch.empty(wl.B, wl.vocab, dtype=torch.float32, device="cuda")
    ws = api.workspace(api.stack_decode_workspace_bytes(st, wl.B), "cuda")
    api.stack_decode(st, torch.from_numpy(tokens).cuda(), torch.from_numpy(pos).cuda(), logits, cos, sin, caches, ws)
    assert api.device_status() == 0
    ref, _ = _stack_decode_reference(wl, layers_st, caches_st, glob, tokens, pos)
    assert_close(f64(logits), ref, TOL["f32"], "fp32 stack decode logits")


def test_stack_decode_graph_replay_matches_direct_calls(api):
    # two consecutive decode steps (positions p, then p + 1 with new tokens written into the
    # same buffers): the replayed graph and direct calls give identical logits and caches
    base = synth.WORKLOADS["stack32_gqa8b_bf16_s8192_v32000"]
    wl = synth.scaled(base, kind="decode", d_model=256, n_heads=8, n_kv_heads=2, d_inter=384, B=4, S=1,
                      T_max=200, pos_lo=0, pos_hi=200, vocab=512, n_layers=2, name="stack2_decode_graph")
    st, caches, _, _, _, tokens, pos = _stack_decode_setup(api, wl, [3, 50, 100, 190])
    caches = [(k.nan_to_num(0.0), v.nan_to_num(0.0)) for k, v in caches]
    twin = [(k.clone(), v.clone()) for k, v in caches]
    cos, sin, _, _ = tables(wl.layer, wl.T_max, oracle)
    tok_d = torch.from_numpy(tokens).cuda()
    pos_d = torch.from_numpy(pos).cuda()
    logits_g = torch.empty(wl.B, wl.vocab, dtype=torch.float32, device="cuda")
    logits_d = torch.empty_like(logits_g)
    ws_g = api.workspace(api.stack_decode_workspace_bytes(st, wl.B), "cuda")
    ws_d = api.workspace(api.stack_decode_workspace_bytes(st, wl.B), "cuda")
    graph = api.StackDecodeGraph(st, tok_d, pos_d, logits_g, cos, sin, caches, ws_g)
    assert graph.kernel_count > 0
    tok2 = torch.from_numpy((tokens * 7 + 3) % wl.vocab).to(torch.int32).cuda()
    for step in range(2):
        if step == 1:
            tok_d.copy_(tok2)
            pos_d.add_(1)
        graph.launch()
        api.stack_decode(st, tok_d, pos_d, logits_d, cos, sin, twin, ws_d)
        torch.cuda.synchronize()
        assert api.device_status() == 0
        assert torch.equal(logits_g, logits_d), f"step {step}"
        for (kg, vg), (kd, vd) in zip(caches, twin):
            assert torch.equal(kg, kd) and torch.equal(vg, vd)
    graph.close()


def _layer_stream(wl, on_layer=None, window=6):
    """Yields each layer's fp64 weights in order, drawn by a pool of spawned processes
    (a bounded number ahead); `on_layer` also receives the storage-format weights."""
    import concurrent.futures as cf
    import multiprocessing as mp
    from gpu_util import gen_layer
    with cf.ProcessPoolExecutor(max_workers=min(16, os.cpu_count() or 4), mp_context=mp.get_context("spawn")) as ex:
        pending = [ex.submit(gen_layer, (wl, l)) for l in range(min(window, wl.n_layers))]
        for l in range(wl.n_layers):
            st = pending.pop(0).result()
            if l + window < wl.n_layers:
                pending.append(ex.submit(gen_layer, (wl, l + window)))
            if on_layer is not None:
                on_layer(st)
            yield {k: v.f64() for k, v in st.items()}


# After 32 bf16 layers, run free from the embedding, the GPU's logits sit some distance from the
# exact oracle's: every layer's bf16 storage roundings cascade (tests/numerics_model.py), and a
# correct implementation cannot follow the oracle's roundings exactly.  That distance is reported
# (the parity log and the printed line), not gated: the gate is the step-by-step check of layers
# 0, 15 and 31 of the same stack on the GPU's own data (test_gpu_teacher_forced.py).  The bound
# below only catches a gross failure (a wrong layer count, a layer skipped, garbage logits).
FREE_RUNNING_SANITY = {"normwise": 0.1}


def test_stack_full_size_causal_prefix(api):
    # the GPU runs all 32 layers on 8192 tokens; logits of the first 64 tokens depend only on
    # those tokens (causality), so the oracle's 64-token run is their reference
    from gpu_util import deviation
    wl = synth.WORKLOADS["stack32_gqa8b_bf16_s8192_v32000"]
    L = wl.layer
    prefix = 64
    glob = synth.stack_globals(wl)
    cos, sin, c64, s64 = tables(L, wl.S, oracle)
    kw = dict(store_bf16=True, **oracle_kw(L))
    tokens = glob["tokens"][:, :prefix]
    g64 = (glob["final_norm"].f64(), glob["embed"].f64(), glob["lm_head"].f64())
    dev_layers = []
    ref = oracle.stack_forward(tokens, _layer_stream(wl, lambda st: dev_layers.append(
        {k: to_dev(v) for k, v in st.items()})), *g64, c64, s64, **kw)
    st = api.StackArgs(dims_of(L), dev_layers, to_dev(glob["final_norm"]), to_dev(glob["embed"]),
                       to_dev(glob["lm_head"]))
    logits = torch.empty(wl.B, wl.S, wl.vocab, dtype=torch.float32, device="cuda")
    ws = api.workspace(st.workspace_bytes(wl.B, wl.S), "cuda")
    api.stack_forward(st, torch.from_numpy(glob["tokens"]).cuda(), logits, cos, sin, ws)
    assert api.device_status() == 0
    gpu = f64(logits[:, :prefix])
    assert np.all(np.isfinite(f64(logits))), "non-finite logits"
    dg = deviation(gpu, ref)
    print(f"stack32 logits, free-running from the embedding: GPU vs oracle {dg}")
    gpu_util.PARITY_LOG.append(("stack32 forward logits, free-running (first 64 rows)", dg["max"], dg["p99"],
                                f"reported; normwise {dg['normwise']:.2e}, sanity bound {FREE_RUNNING_SANITY}"))
    assert dg["normwise"] <= FREE_RUNNING_SANITY["normwise"], dg


def test_stack_decode_full_size_sampled(api):
    # the bench's 32-layer decode step: 64 sequences with 4096-slot caches in every layer.  The
    # GPU runs all of them; the oracle follows two through the 32 layers (weights streamed layer
    # by layer).  The free-running distance is reported as for the stack forward above.
    from gpu_util import deviation
    wl = synth.WORKLOADS["stack32_decode_gqa8b_bf16_b64_t4096_v32000"]
    L = wl.layer
    B, T = wl.B, wl.T_max
    sample = [3, 41]
    glob = synth.stack_globals(wl)
    tokens = glob["tokens"][:, 0].copy()
    pos = synth.decode_positions(wl)
    pmax = int(pos[sample].max())
    cos, sin, c64, s64 = tables(L, T, oracle)
    kw = dict(store_bf16=True, **oracle_kw(L))
    g = torch.Generator(device="cuda").manual_seed(wl.seed)
    dev_layers, caches, sampled = [], [], []

    def on_layer(st):
        dev_layers.append({k: to_dev(v) for k, v in st.items()})
        k = torch.empty(B, L.n_kv_heads, T, L.head_dim, dtype=torch.bfloat16, device="cuda").normal_(generator=g)
        v = torch.empty_like(k).normal_(generator=g)
        caches.append((k, v))
        sampled.append((f64(k[sample, :, :pmax]), f64(v[sample, :, :pmax])))

    x = glob["embed"].f64()[tokens[sample]][:, None, :]
    for l, w64 in enumerate(_layer_stream(wl, on_layer)):
        pk, pv = sampled[l]
        x, _, _ = oracle.decoder_layer(x, w64, c64, s64, past_k=pk, past_v=pv, past_len=pos[sample], **kw)
        x = oracle.round_bf16(x)
    xn = oracle.round_bf16(oracle.rms_norm(x[:, 0], glob["final_norm"].f64(), L.rms_eps))
    ref = xn @ glob["lm_head"].f64().T
    st = api.StackArgs(dims_of(L), dev_layers, to_dev(glob["final_norm"]), to_dev(glob["embed"]),
                       to_dev(glob["lm_head"]))
    logits = torch.empty(B, wl.vocab, dtype=torch.float32, device="cuda")
    ws = api.workspace(api.stack_decode_workspace_bytes(st, B), "cuda")
    api.stack_decode(st, torch.from_numpy(tokens).cuda(), torch.from_numpy(pos).cuda(), logits, cos, sin, caches, ws)
    assert api.device_status() == 0
    assert torch.isfinite(logits).all(), "non-finite logits"
    dg = deviation(f64(logits[sample]), ref)
    print(f"stack32 decode logits, free-running: GPU vs oracle {dg}")
    gpu_util.PARITY_LOG.append(("stack32 decode logits, free-running (sequences 3, 41)", dg["max"], dg["p99"],
                                f"reported; normwise {dg['normwise']:.2e}, sanity bound {FREE_RUNNING_SANITY}"))
    assert dg["normwise"] <= FREE_RUNNING_SANITY["normwise"], dg
