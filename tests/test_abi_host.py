"""Host-side checks of the C ABI: the library builds and loads, exports every symbol the
header declares, and rejects bad arguments before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from conftest import ROOT


@pytest.fixture(scope="module")
def native():
    from llama_decoder_block_gb300 import build, _native
    build.build()
    return _native


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "llama_layer.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(llama_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("llama_layer_prefill", "llama_layer_decode", "llama_stack_forward", "llama_rope_tables",
                     "llama_get_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(native):
    lib = ctypes.CDLL(native.LIB_PATH)
    names = _declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding declares exactly the header's functions
    assert sorted(native.SIGNATURES) == names


def test_rope_tables_match_the_oracle(native):
    from llama_decoder_block_gb300 import api
    for base, D, P in ((1e4, 16, 64), (5e5, 128, 4096), (1e4, 128, 2048)):
        cos, sin = api.rope_tables(base, D, P)
        oc, os_ = oracle.rope_tables(base, D, P)
        # both round an fp64 value to fp32; allow one fp32 ulp for libm differences
        assert np.max(np.abs(cos - oc.astype(np.float32))) <= 2 ** -24
        assert np.max(np.abs(sin - os_.astype(np.float32))) <= 2 ** -24


def test_status_strings(native):
    lib = native.lib()
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.llama_status_string(code)
    assert lib.llama_status_string(-99) == b"unknown status"


def _dims(native, **kw):
    base = dict(d_model=256, n_heads=4, n_kv_heads=2, head_dim=128, d_inter=384, rms_eps=1e-5, dtype=1)
    base.update(kw)
    return native.LayerDims(**base)


def _bytes(native, dims, B=2, S=64):
    n = ctypes.c_size_t()
    rc = native.lib().llama_layer_prefill_workspace_bytes(ctypes.byref(dims), B, S, ctypes.byref(n))
    return rc, n.value


def test_workspace_sizes_and_dims_validation(native):
    rc, n = _bytes(native, _dims(native))
    assert rc == 0 and n >= 2 * 2 * 64 * (2 * 256 + 2 * 512 + 384)   # xn, h, q, o, a
    assert _bytes(native, _dims(native, n_kv_heads=3))[0] == -1     # H % G != 0
    assert _bytes(native, _dims(native, head_dim=15, dtype=0))[0] == -1   # odd D
    assert _bytes(native, _dims(native, head_dim=64))[0] == -2      # bf16 tile path needs D = 128
    assert _bytes(native, _dims(native, d_model=200))[0] == -2      # d % 128
    assert _bytes(native, _dims(native, dtype=7))[0] == -1
    assert _bytes(native, _dims(native, rms_eps=-1.0))[0] == -1
    assert _bytes(native, _dims(native, n_heads=12, n_kv_heads=4))[0] == -2   # H/G = 3 not a tiled ratio
    assert _bytes(native, _dims(native, n_heads=24, n_kv_heads=2))[0] == -2   # H/G = 12: not 1, 2, 4 or 8k
    assert _bytes(native, _dims(native, n_heads=32, n_kv_heads=1))[0] == 0    # MQA: query heads in groups of 8
    assert _bytes(native, _dims(native, rope_style=1))[0] == 0               # half-split RoPE pairs
    assert _bytes(native, _dims(native, rope_style=2))[0] == -1
    assert _bytes(native, _dims(native, head_dim=16, d_model=64, n_heads=4, n_kv_heads=2, d_inter=176,
                                dtype=0))[0] == 0                     # the fp32 path takes any even D


def test_prefill_rejects_bad_arguments_without_a_gpu(native):
    lib = native.lib()
    dims = _dims(native)
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.addressof(buf)
    p = (p + 255) // 256 * 256 - 256 + 256 if p % 256 else p
    w = native.LayerWeights(*([p] * 9))
    cache = native.KVCache(p, p, 64)

    def call(dims=dims, w=w, x=p, out=p + 1024, cos=p, sin=p, max_pos=64, cache=cache, B=1, S=8, ws=p, n=1 << 40):
        return lib.llama_layer_prefill(ctypes.byref(dims), ctypes.byref(w), x, out, cos, sin, max_pos, cache, B, S,
                                       ws, n, None)

    assert call(x=None) == -1
    assert call(out=p) == -1                   # aliasing input and output
    assert call(x=p + 8) == -1                 # not 16-byte aligned
    assert call(S=65) == -1                    # S > max_T
    assert call(max_pos=4) == -1               # S > max_pos
    assert call(n=16) == -1                    # workspace too small
    assert call(B=0) == -1
    assert call(w=native.LayerWeights(*([p] * 8 + [None]))) == -1
    assert call(dims=_dims(native, n_kv_heads=3)) == -1


def test_decode_and_attention_reject_bad_arguments_without_a_gpu(native):
    lib = native.lib()
    dims = _dims(native)
    buf = (ctypes.c_uint8 * 4096)()
    p = (ctypes.addressof(buf) + 255) // 256 * 256
    w = native.LayerWeights(*([p] * 9))
    cache = native.KVCache(p, p, 64)
    assert lib.llama_layer_decode(ctypes.byref(dims), ctypes.byref(w), p, p + 512, p, p, 64, None, cache, 1, p, 1 << 30,
                                  None) == -1
    assert lib.llama_layer_decode(ctypes.byref(dims), ctypes.byref(w), p, p, p, p, 64, p, cache, 1, p, 1 << 30,
                                  None) == -1
    assert lib.llama_attention_prefill(ctypes.byref(dims), p, native.KVCache(p, p, 4), p, 1, 8, None) == -1
    assert lib.llama_linear_bf16(p, p, p, 4, 12, 30, 0, None) == -2    # K % 8
    assert lib.llama_linear_bf16(None, p, p, 4, 16, 32, 0, None) == -1
    assert lib.llama_rmsnorm(p, p, p, 4, 64, -1.0, 1, None) == -1
    assert lib.llama_layernorm(p, p, None, p, 4, 64, 1e-5, 1, None) == -1
    assert lib.llama_layernorm(p, p, p + 8, p, 4, 64, 1e-5, 1, None) == -1     # beta not 16-byte aligned
    assert lib.llama_layernorm(p, p, p, p, 4, 64, 1e-5, 7, None) == -1        # unknown dtype
    assert lib.llama_rope_tables(1e4, 7, 4, p, p) == -1


def test_workspace_layout_names_disjoint_regions_inside_the_workspace(native):
    lib = native.lib()
    for dt in (0, 1):
        dims = _dims(native, dtype=dt)
        B, S = 2, 64
        offs = (ctypes.c_size_t * 5)()
        assert lib.llama_layer_prefill_workspace_layout(ctypes.byref(dims), B, S, offs) == 0
        rc, total = _bytes(native, dims, B, S)
        assert rc == 0
        es = 2 if dt == 1 else 4
        sizes = [B * 4 * S * 128 * es, B * S * 4 * 128 * es, B * S * 256 * es, B * S * 384 * es,
                 B * S * 256 * es]                                                         # q, o, h, a, hn
        spans = sorted((o, o + n) for o, n in zip(offs, sizes))
        assert all(o % 256 == 0 for o in offs)
        assert all(a_end <= b_start for (_, a_end), (b_start, _) in zip(spans, spans[1:]))
        assert spans[-1][1] <= total
    assert lib.llama_layer_prefill_workspace_layout(ctypes.byref(_dims(native)), 2, 64, None) == -1
    assert lib.llama_layer_prefill_workspace_layout(ctypes.byref(_dims(native, n_kv_heads=3)), 2, 64, offs) == -1


def test_norm_fused_steps_reject_bad_arguments_without_a_gpu(native):
    lib = native.lib()
    buf = (ctypes.c_uint8 * 8192)()
    p = (ctypes.addressof(buf) + 255) // 256 * 256
    xn, sy = p + 4096, p + 2048
    assert lib.llama_norm_linear_bf16(p, p, 1e-5, p, p, 4, 16, 60, 0, xn, sy, None) == -2       # K % 8
    assert lib.llama_norm_linear_bf16(p, None, 1e-5, p, p, 4, 16, 64, 0, xn, sy, None) == -1    # no gamma
    assert lib.llama_norm_linear_bf16(p, p, 1e-5, p, p, 4, 16, 64, 0, None, sy, None) == -1     # no xn
    assert lib.llama_norm_linear_bf16(p, p, 1e-5, p, p, 4, 16, 64, 0, xn, None, None) == -1     # no sync
    assert lib.llama_norm_linear_bf16(p, p, 1e-5, p, p, 4, 16, 64, 0, p, sy, None) == -1        # xn aliases A
    assert lib.llama_norm_linear_bf16(p, p, -1.0, p, p, 4, 16, 64, 0, xn, sy, None) == -1       # eps < 0
    assert lib.llama_norm_linear_bf16(p, p + 8, 1e-5, p, p, 4, 16, 64, 0, xn, sy, None) == -1   # gamma misaligned
    assert lib.llama_norm_linear_swiglu(p, p, 1e-5, p, p, p, 4, 96, 64, xn, sy, None) == -2     # I % 128
    assert lib.llama_norm_linear_swiglu(p, p, 1e-5, p, p, None, 4, 128, 64, xn, sy, None) == -1
    dims = _dims(native)
    cache = native.KVCache(p, p, 64)
    call = lambda **kw: lib.llama_norm_qkv_rope(ctypes.byref(kw.get("dims", dims)), p, kw.get("g", p), p, p, p, p, p,
                                                kw.get("max_pos", 64), cache, p, 1, kw.get("S", 8), kw.get("xn", xn),
                                                sy, None)
    assert call(g=None) == -1
    assert call(xn=None) == -1
    assert call(S=65) == -1                      # S > max_T
    assert call(max_pos=4) == -1                 # S > max_pos
    assert call(dims=_dims(native, head_dim=16, d_model=64, n_heads=4, n_kv_heads=2, d_inter=176, dtype=0)) == -2
