"""Each step of the bf16 layer at the full sizes of the benchmark workloads, through the C ABI.

The GPU runs every step over all rows in the launch shape the benchmark uses; the oracle
recomputes sampled rows (GEMM rows are independent, attention rows need only their own keys).
One step at a time there is a single bf16 rounding between oracle and GPU, so the bf16
tolerance 2e-2 * (1 + |ref|) holds elementwise, and so does the tighter one-ulp bound below.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, assert_close, bf16_stored, dims_of, f64, tables, to_dev
from llama_decoder_block_gb300 import synth

pytestmark = pytest.mark.gpu

FULL = ["mha7b_bf16_b1_s2048", "gqa8b_bf16_b4_s4096"]


@pytest.fixture(scope="module")
def api(cuda_dev):
    from llama_decoder_block_gb300 import build, api as a
    build.build()
    assert a.device_status() == 0
    return a


def _rows(M, S, n=160, seed=0):
    rng = np.random.default_rng(seed)
    r = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    r |= {0, M - 1, S - 1} | {b * S for b in range(M // S)}
    return np.array(sorted(r))


def _one_ulp(gpu, ref, what):
    """bf16 output of an fp32-accumulated result: within one bf16 ulp (2^-8 relative) plus
    the accumulation error, which 1e-3 of the row's rms bounds generously."""
    scale = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bad = np.abs(gpu - ref) > 2.0 ** -8 * np.abs(ref) + 1e-3 * scale
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond one bf16 ulp, first at {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("name", FULL)
def test_steps_full_size(api, name):
    wl = synth.WORKLOADS[name]
    L = wl.layer
    B, S, d, H, G, D, I = wl.B, wl.S, L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter
    M = B * S
    st = synth.layer_weights(wl)
    w = {k: to_dev(v) for k, v in st.items()}
    w64 = {k: v.f64() for k, v in st.items()}
    rng = np.random.default_rng(99)
    rows = _rows(M, S)
    dims = dims_of(L)
    tol = TOL["bf16"]

    # a1 / a6: RMSNorm
    xs = synth.activations(wl)
    x = to_dev(xs).view(M, d)
    xn = torch.empty_like(x)
    api.rmsnorm(x, w["attn_norm"], xn, L.rms_eps)
    x64 = xs.f64().reshape(M, d)
    ref = oracle.rms_norm(x64[rows], w64["attn_norm"], L.rms_eps)
    assert_close(f64(xn)[rows], ref, tol, "rmsnorm")
    _one_ulp(f64(xn)[rows], ref, "rmsnorm")

    # a2 + a3: QKV projection with RoPE, k and v scattered into the cache
    xin = bf16_stored(rng.standard_normal((M, d)))
    q = torch.empty(B, H, S, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.empty(B, G, S, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    cos, sin, c64, s64 = tables(L, S, oracle)
    api.qkv_rope(dims, to_dev(xin).view(B, S, d), w["wq"], w["wk"], w["wv"], cos, sin, kc, vc, q)
    xin64 = xin.f64()[rows]
    b_of, s_of = rows // S, rows % S
    q_ref = oracle.apply_rope(oracle.linear(xin64, w64["wq"]).reshape(-1, H, D), c64[s_of][:, None], s64[s_of][:, None])
    k_ref = oracle.apply_rope(oracle.linear(xin64, w64["wk"]).reshape(-1, G, D), c64[s_of][:, None], s64[s_of][:, None])
    v_ref = oracle.linear(xin64, w64["wv"]).reshape(-1, G, D)
    q_gpu = f64(q)[b_of, :, s_of]
    assert_close(q_gpu, q_ref, tol, "qkv: q")
    assert_close(f64(kc)[b_of, :, s_of], k_ref, tol, "qkv: k in cache")
    assert_close(f64(vc)[b_of, :, s_of], v_ref, tol, "qkv: v in cache")
    _one_ulp(q_gpu, q_ref, "qkv: q")

    # a4: causal GQA attention over the whole cache
    qs = bf16_stored(rng.standard_normal((B, H, S, D)))
    ks = bf16_stored(rng.standard_normal((B, G, S, D)))
    vs = bf16_stored(rng.standard_normal((B, G, S, D)))
    o = torch.empty(B, S, H * D, dtype=torch.bfloat16, device="cuda")
    api.attention_prefill(dims, to_dev(qs), to_dev(ks), to_dev(vs), o)
    o_h = f64(o).reshape(B, S, H, D)
    for b, i in zip(b_of, s_of):
        for h in rng.choice(H, size=4, replace=False):
            ref = oracle.attention(qs.f64()[b:b + 1, h:h + 1, i:i + 1], ks.f64()[b:b + 1, h // (H // G):h // (H // G) + 1, :i + 1],
                                   vs.f64()[b:b + 1, h // (H // G):h // (H // G) + 1, :i + 1], np.array([[i]]),
                                   np.array([i + 1]))[0, 0, 0]
            assert_close(o_h[b, i, h], ref, tol, f"attention b={b} i={i} h={h}")

    # a5: o_proj + residual
    oin = bf16_stored(0.6 * rng.standard_normal((M, H * D)))
    h_out = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    api.linear_residual(to_dev(oin), w["wo"], x, h_out)
    ref = x64[rows] + oracle.linear(oin.f64()[rows], w64["wo"])
    assert_close(f64(h_out)[rows], ref, tol, "o_proj + residual")
    _one_ulp(f64(h_out)[rows], ref, "o_proj + residual")

    # a7: gate/up + SiLU * up
    hn = bf16_stored(rng.standard_normal((M, d)))
    a = torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
    api.linear_swiglu(to_dev(hn), w["w_gate"], w["w_up"], a)
    hn64 = hn.f64()[rows]
    ref = oracle.silu(oracle.linear(hn64, w64["w_gate"])) * oracle.linear(hn64, w64["w_up"])
    assert_close(f64(a)[rows], ref, tol, "gate/up SwiGLU")
    _one_ulp(f64(a)[rows], ref, "gate/up SwiGLU")

    # a8: down + residual
    ain = bf16_stored(rng.standard_normal((M, I)))
    out = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    api.linear_residual(to_dev(ain), w["w_down"], x, out)
    ref = x64[rows] + oracle.linear(ain.f64()[rows], w64["w_down"])
    assert_close(f64(out)[rows], ref, tol, "down + residual")
    _one_ulp(f64(out)[rows], ref, "down + residual")
    assert api.device_status() == 0


def test_decode_layer_back_to_back_calls_finish_cleanly(api):
    # 1500 decode steps of the full-size layer queued without a host synchronisation between
    # them: the kernels overlap each other's tails, so any barrier that a fast producer could
    # run two phases ahead of its consumer would stall a wait here (LLAMA_ERR_TIMEOUT)
    wl = synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"]
    L = wl.layer
    B, T = wl.B, wl.T_max
    g = torch.Generator(device="cuda").manual_seed(11)
    d, H, G, D, I = L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter
    shapes = {"wq": (H * D, d), "wk": (G * D, d), "wv": (G * D, d), "wo": (d, H * D), "w_gate": (I, d),
              "w_up": (I, d), "w_down": (d, I)}
    w = {k: (torch.randn(s, generator=g, device="cuda") * 0.02).to(torch.bfloat16) for k, s in shapes.items()}
    w["attn_norm"] = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    w["ffn_norm"] = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    kc = torch.randn(B, G, T, D, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn_like(kc)
    pos = torch.from_numpy(synth.decode_positions(wl)).cuda()
    x = torch.randn(B, d, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(x)
    cos, sin, _, _ = tables(L, T, oracle)
    dims = dims_of(L)
    ws = api.workspace(api.decode_workspace_bytes(dims, B, T), "cuda")
    for _ in range(15):
        for _ in range(100):
            api.layer_decode(dims, w, x, out, cos, sin, pos, kc, vc, ws)
        rc = api.device_status()
        assert rc == 0, (rc, api.timeout_record())
    assert torch.isfinite(out.float()).all()
