"""Seeded synthetic inputs for the decoder-layer workloads.

This module only draws random numbers and converts them to their storage
formats (fp32, bf16 bit patterns, int32).  It holds none of the layer's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Recipe (every tensor has its own PCG64 stream keyed by
``(seed, layer, tensor_id)``, so any tensor can be regenerated alone):

* activations ``x`` ~ N(0, 1);
* linear weights ~ N(0, 0.02), ``nn.Linear`` layout ``[out, in]``, no bias
  (page "12 · 从 Transformer 到 LLaMA 系列", §八 ``_init_weights``);
* RMSNorm gamma: all ones (same page, §八 ``RMSNorm.__init__``) or
  1 + N(0, 0.1) where the workload says so;
* embedding table ~ N(0, 0.02), tokens uniform in [0, vocab);
* decode: cache K/V ~ N(0, 1), positions uniform in [lo, hi).

Draws are fp32 (fp64 for the fp32 workload) and are rounded once, to nearest
even, to the storage type.
"""
from __future__ import annotations

import dataclasses
import numpy as np

# tensor ids of the per-tensor streams
_X, _ATTN_NORM, _WQ, _WK, _WV, _WO, _FFN_NORM, _WGATE, _WUP, _WDOWN = range(10)
_EMBED, _LM_HEAD, _TOKENS, _POSITIONS, _CACHE_K, _CACHE_V, _FINAL_NORM = range(10, 17)

LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


@dataclasses.dataclass(frozen=True)
class LayerShape:
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_inter: int
    rms_eps: float
    rope_base: float
    dtype: str            # "f32" or "bf16"
    gamma: str            # "ones" or "noisy" (1 + N(0, 0.1))
    rope_style: str = "even_odd"   # or "half": RoPE pairs (i, i + D/2)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str             # "prefill", "decode" or "stack"
    layer: LayerShape
    seed: int
    B: int
    S: int = 0            # prefill / stack sequence length
    T_max: int = 0        # decode: cache capacity per sequence
    pos_lo: int = 0       # decode: new-token positions uniform in [pos_lo, pos_hi)
    pos_hi: int = 0
    n_layers: int = 1
    vocab: int = 0


TINY_LAYER = LayerShape(64, 4, 2, 16, 176, 1e-5, 1e4, "f32", "ones")
MHA_7B_LAYER = LayerShape(4096, 32, 32, 128, 11008, 1e-6, 1e4, "bf16", "noisy")
GQA_8B_LAYER = LayerShape(4096, 32, 8, 128, 14336, 1e-5, 5e5, "bf16", "noisy")
GQA_8B_LAYER_INIT = dataclasses.replace(GQA_8B_LAYER, gamma="ones")

WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_f32_b1_s16", "prefill", TINY_LAYER, 1001, B=1, S=16),
        Workload("mha7b_bf16_b1_s2048", "prefill", MHA_7B_LAYER, 1002, B=1, S=2048),
        Workload("gqa8b_bf16_b4_s4096", "prefill", GQA_8B_LAYER, 1003, B=4, S=4096),
        Workload("decode_gqa8b_bf16_b64_t4096", "decode", GQA_8B_LAYER, 1004, B=64,
                 T_max=4096, pos_lo=1024, pos_hi=4096),
        Workload("stack32_gqa8b_bf16_s8192_v32000", "stack", GQA_8B_LAYER_INIT, 1005, B=1,
                 S=8192, n_layers=32, vocab=32000),
        # one decode step of that 32-layer model for the decode workload's 64 sequences
        Workload("stack32_decode_gqa8b_bf16_b64_t4096_v32000", "decode", GQA_8B_LAYER_INIT, 1006, B=64,
                 S=1, T_max=4096, pos_lo=1024, pos_hi=4096, n_layers=32, vocab=32000),
    )
}


def rng(seed: int, layer: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, tensor_id])))


# ---------------------------------------------------------------- storage formats

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to nearest-even bf16; returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    r = np.where(nan, np.uint32(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Stored:
    """A tensor in its storage format: ``data`` is float32, or uint16 bf16 bits."""
    data: np.ndarray
    dtype: str

    @property
    def shape(self):
        return self.data.shape

    def f64(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.data).astype(np.float64)
        return self.data.astype(np.float64)


def _store(vals: np.ndarray, dtype: str) -> Stored:
    if dtype == "bf16":
        return Stored(f32_to_bf16_bits(vals.astype(np.float32, copy=False)), "bf16")
    return Stored(np.ascontiguousarray(vals, dtype=np.float32), "f32")


def _normal(g: np.random.Generator, shape, std: float, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return g.standard_normal(shape) * std                      # fp64 draws
    v = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return v


# ---------------------------------------------------------------- generators

def layer_weights(wl: Workload, layer: int = 0) -> dict[str, Stored]:
    L = wl.layer
    d, H, G, D, I = L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter
    shapes = {
        "wq": ((H * D, d), _WQ), "wk": ((G * D, d), _WK), "wv": ((G * D, d), _WV),
        "wo": ((d, H * D), _WO), "w_gate": ((I, d), _WGATE), "w_up": ((I, d), _WUP),
        "w_down": ((d, I), _WDOWN),
    }
    out = {}
    for name, tid in (("attn_norm", _ATTN_NORM), ("ffn_norm", _FFN_NORM)):
        if L.gamma == "ones":
            out[name] = _store(np.ones(d), L.dtype)
        else:
            out[name] = _store(1.0 + _normal(rng(wl.seed, layer, tid), (d,), 0.1, L.dtype), L.dtype)
    for name, (shape, tid) in shapes.items():
        out[name] = _store(_normal(rng(wl.seed, layer, tid), shape, 0.02, L.dtype), L.dtype)
    return {k: out[k] for k in LAYER_TENSORS}


def activations(wl: Workload, rows: int | None = None) -> Stored:
    """x: ``[B, S, d]`` for prefill, ``[B, d]`` (one new token each) for decode."""
    L = wl.layer
    shape = (wl.B, wl.S, L.d_model) if wl.kind == "prefill" else (wl.B, L.d_model)
    return _store(_normal(rng(wl.seed, 0, _X), shape, 1.0, L.dtype), L.dtype)


def decode_positions(wl: Workload) -> np.ndarray:
    """New-token positions ``[B]`` int32, uniform in [pos_lo, pos_hi)."""
    return rng(wl.seed, 0, _POSITIONS).integers(wl.pos_lo, wl.pos_hi, size=wl.B).astype(np.int32)


def decode_state(wl: Workload, layer: int = 0) -> tuple[np.ndarray, Stored, Stored]:
    """positions ``[B]`` int32 and layer ``layer``'s pre-filled caches K, V ``[B, G, T_max, D]``."""
    L = wl.layer
    pos = decode_positions(wl)
    shape = (wl.B, L.n_kv_heads, wl.T_max, L.head_dim)
    k = _store(_normal(rng(wl.seed, layer, _CACHE_K), shape, 1.0, L.dtype), L.dtype)
    v = _store(_normal(rng(wl.seed, layer, _CACHE_V), shape, 1.0, L.dtype), L.dtype)
    return pos, k, v


def stack_globals(wl: Workload) -> dict[str, Stored | np.ndarray]:
    """tokens ``[B, S]``, embedding ``[V, d]``, untied LM head ``[V, d]``, final-norm gamma."""
    L = wl.layer
    tokens = rng(wl.seed, 0, _TOKENS).integers(0, wl.vocab, size=(wl.B, wl.S)).astype(np.int32)
    embed = _store(_normal(rng(wl.seed, 0, _EMBED), (wl.vocab, L.d_model), 0.02, L.dtype), L.dtype)
    lm_head = _store(_normal(rng(wl.seed, 0, _LM_HEAD), (wl.vocab, L.d_model), 0.02, L.dtype), L.dtype)
    final_norm = _store(np.ones(L.d_model), L.dtype)
    return {"tokens": tokens, "embed": embed, "lm_head": lm_head, "final_norm": final_norm}


def scaled(wl: Workload, **changes) -> Workload:
    """The same workload recipe at other sizes (parity cases that the oracle finishes quickly)."""
    layer_changes = {k: changes.pop(k) for k in list(changes) if k in LayerShape.__dataclass_fields__}
    layer = dataclasses.replace(wl.layer, **layer_changes) if layer_changes else wl.layer
    name = changes.pop("name", wl.name + "_scaled")
    return dataclasses.replace(wl, layer=layer, name=name, **changes)
