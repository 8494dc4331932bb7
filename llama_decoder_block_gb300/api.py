"""Thin Python binding of the C ABI: torch tensors in, device pointers out.

Every step runs in the library's CUDA kernels; this module only builds the argument
structs, sizes workspaces and turns status codes into exceptions.  PyTorch provides
device memory and streams.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import _native as N

DTYPES = {torch.float32: N.LLAMA_F32, torch.bfloat16: N.LLAMA_BF16}


@dataclass(frozen=True)
class Dims:
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_inter: int
    rms_eps: float
    dtype: torch.dtype
    rope_style: int = 0     # 0: pairs (2i, 2i+1); 1: pairs (i, i + D/2)

    def c(self) -> N.LayerDims:
        return N.LayerDims(self.d_model, self.n_heads, self.n_kv_heads, self.head_dim, self.d_inter,
                           self.rms_eps, DTYPES[self.dtype], self.rope_style)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def weights_struct(w: dict) -> N.LayerWeights:
    return N.LayerWeights(*[_ptr(w[k]) for k in N.WEIGHT_FIELDS])


def cache_struct(k: torch.Tensor, v: torch.Tensor) -> N.KVCache:
    return N.KVCache(_ptr(k), _ptr(v), k.shape[2])


def rope_tables(base: float, head_dim: int, max_pos: int) -> tuple[np.ndarray, np.ndarray]:
    """Host cos/sin tables [max_pos, head_dim/2] fp32 (llama_rope_tables)."""
    cos = np.empty((max_pos, head_dim // 2), dtype=np.float32)
    sin = np.empty_like(cos)
    N.check(N.lib().llama_rope_tables(base, head_dim, max_pos, cos.ctypes.data, sin.ctypes.data), "llama_rope_tables")
    return cos, sin


def prefill_workspace_bytes(dims: Dims, B: int, S: int) -> int:
    n = ctypes.c_size_t()
    d = dims.c()
    N.check(N.lib().llama_layer_prefill_workspace_bytes(ctypes.byref(d), B, S, ctypes.byref(n)), "workspace")
    return n.value


def decode_workspace_bytes(dims: Dims, B: int, max_T: int) -> int:
    n = ctypes.c_size_t()
    d = dims.c()
    N.check(N.lib().llama_layer_decode_workspace_bytes(ctypes.byref(d), B, max_T, ctypes.byref(n)), "workspace")
    return n.value


def workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def layer_prefill(dims: Dims, w: dict, x, out, cos, sin, cache_k, cache_v, ws, stream=None) -> None:
    B, S = x.shape[0], x.shape[1]
    d = dims.c()
    ww = weights_struct(w)
    N.check(N.lib().llama_layer_prefill(ctypes.byref(d), ctypes.byref(ww), _ptr(x), _ptr(out), _ptr(cos), _ptr(sin),
                                        cos.shape[0], cache_struct(cache_k, cache_v), B, S, _ptr(ws), ws.numel(),
                                        _stream(stream)), "llama_layer_prefill")


def layer_prefill_chunk(dims: Dims, w: dict, x, out, cos, sin, start, cache_k, cache_v, ws, lengths=None,
                        stream=None) -> None:
    """A chunk of S tokens per sequence on top of the cache: token s of sequence b at position
    start[b] + s (start, lengths: device int32 [B]; lengths None = all S)."""
    B, S = x.shape[0], x.shape[1]
    d = dims.c()
    ww = weights_struct(w)
    N.check(N.lib().llama_layer_prefill_chunk(ctypes.byref(d), ctypes.byref(ww), _ptr(x), _ptr(out), _ptr(cos),
                                              _ptr(sin), cos.shape[0], _ptr(start), _ptr(lengths),
                                              cache_struct(cache_k, cache_v), B, S, _ptr(ws), ws.numel(),
                                              _stream(stream)), "llama_layer_prefill_chunk")


def layer_decode(dims: Dims, w: dict, x, out, cos, sin, positions, cache_k, cache_v, ws, stream=None) -> None:
    d = dims.c()
    ww = weights_struct(w)
    N.check(N.lib().llama_layer_decode(ctypes.byref(d), ctypes.byref(ww), _ptr(x), _ptr(out), _ptr(cos), _ptr(sin),
                                       cos.shape[0], _ptr(positions), cache_struct(cache_k, cache_v), x.shape[0],
                                       _ptr(ws), ws.numel(), _stream(stream)), "llama_layer_decode")


class StackArgs:
    """Keeps the ctypes structs of a stack alive for as long as it is used."""

    def __init__(self, dims: Dims, layers: list[dict], final_norm, embed, lm_head):
        self.layer_structs = (N.LayerWeights * max(1, len(layers)))(*[weights_struct(w) for w in layers])
        self.tensors = (layers, final_norm, embed, lm_head)
        self.dims = dims
        self.s = N.Stack(len(layers), embed.shape[0], dims.c(), self.layer_structs, _ptr(final_norm), _ptr(embed),
                         _ptr(lm_head))

    def workspace_bytes(self, B: int, S: int) -> int:
        n = ctypes.c_size_t()
        N.check(N.lib().llama_stack_workspace_bytes(ctypes.byref(self.s), B, S, ctypes.byref(n)), "workspace")
        return n.value


def stack_forward(st: StackArgs, tokens, logits, cos, sin, ws, caches=None, stream=None) -> None:
    B, S = tokens.shape
    cache_arr = None
    if caches is not None:
        cache_arr = (N.KVCache * len(caches))(*[cache_struct(k, v) for k, v in caches])
    N.check(N.lib().llama_stack_forward(ctypes.byref(st.s), _ptr(tokens), _ptr(logits), _ptr(cos), _ptr(sin),
                                        cos.shape[0], cache_arr, B, S, _ptr(ws), ws.numel(), _stream(stream)),
            "llama_stack_forward")


def stack_decode_workspace_bytes(st: StackArgs, B: int) -> int:
    n = ctypes.c_size_t()
    N.check(N.lib().llama_stack_decode_workspace_bytes(ctypes.byref(st.s), B, ctypes.byref(n)), "workspace")
    return n.value


def _cache_array(caches):
    return (N.KVCache * max(1, len(caches)))(*[cache_struct(k, v) for k, v in caches])


def stack_decode(st: StackArgs, tokens, positions, logits, cos, sin, caches, ws, stream=None) -> None:
    """One decode step of the stack: tokens, positions [B] int32; caches: list of (k, v)."""
    N.check(N.lib().llama_stack_decode(ctypes.byref(st.s), _ptr(tokens), _ptr(positions), _ptr(logits), _ptr(cos),
                                       _ptr(sin), cos.shape[0], _cache_array(caches), tokens.shape[0], _ptr(ws),
                                       ws.numel(), _stream(stream)), "llama_stack_decode")


class StackDecodeGraph:
    """A decode step of the stack captured once as a CUDA graph and replayed with launch().

    The graph reads the tokens and positions in the given buffers at each replay; every
    tensor passed here must outlive the graph (this object keeps references to them).
    """

    def __init__(self, st: StackArgs, tokens, positions, logits, cos, sin, caches, ws):
        self._keep = (st, tokens, positions, logits, cos, sin, list(caches), ws)
        self._arr = _cache_array(caches)
        h = ctypes.c_void_p()
        N.check(N.lib().llama_stack_decode_graph(ctypes.byref(st.s), _ptr(tokens), _ptr(positions), _ptr(logits),
                                                 _ptr(cos), _ptr(sin), cos.shape[0], self._arr, tokens.shape[0],
                                                 _ptr(ws), ws.numel(), ctypes.byref(h)), "llama_stack_decode_graph")
        self._h = h

    @property
    def kernel_count(self) -> int:
        return N.lib().llama_graph_kernel_count(self._h)

    def launch(self, stream=None) -> None:
        N.check(N.lib().llama_graph_launch(self._h, _stream(stream)), "llama_graph_launch")

    def close(self) -> None:
        if self._h is not None and self._h.value:
            N.lib().llama_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def rmsnorm(x, gamma, y, eps: float, stream=None) -> None:
    d = x.shape[-1]
    N.check(N.lib().llama_rmsnorm(_ptr(x), _ptr(gamma), _ptr(y), x.numel() // d, d, eps, DTYPES[x.dtype],
                                  _stream(stream)), "llama_rmsnorm")


def layernorm(x, gamma, beta, y, eps: float, stream=None) -> None:
    d = x.shape[-1]
    N.check(N.lib().llama_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), x.numel() // d, d, eps,
                                    DTYPES[x.dtype], _stream(stream)), "llama_layernorm")


def linear_bf16(a, b, c, stream=None) -> None:
    M, K = a.shape
    Nn = b.shape[0]
    N.check(N.lib().llama_linear_bf16(_ptr(a), _ptr(b), _ptr(c), M, Nn, K, int(c.dtype == torch.float32),
                                      _stream(stream)), "llama_linear_bf16")


def linear_residual(a, w, resid, out, stream=None) -> None:
    M, K = a.shape
    N.check(N.lib().llama_linear_residual(_ptr(a), _ptr(w), _ptr(resid), _ptr(out), M, w.shape[0], K,
                                          _stream(stream)), "llama_linear_residual")


def linear_swiglu(a, w_gate, w_up, out, stream=None) -> None:
    M, K = a.shape
    N.check(N.lib().llama_linear_swiglu(_ptr(a), _ptr(w_gate), _ptr(w_up), _ptr(out), M, w_gate.shape[0], K,
                                        _stream(stream)), "llama_linear_swiglu")


def qkv_rope(dims: Dims, xn, wq, wk, wv, cos, sin, cache_k, cache_v, q_out, stream=None) -> None:
    B, S = xn.shape[0], xn.shape[1]
    d = dims.c()
    N.check(N.lib().llama_qkv_rope(ctypes.byref(d), _ptr(xn), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(cos), _ptr(sin),
                                   cos.shape[0], cache_struct(cache_k, cache_v), _ptr(q_out), B, S, _stream(stream)),
            "llama_qkv_rope")


def _norm_buffers(rows: int, K: int, like: torch.Tensor, xn, sync):
    if xn is None:
        xn = torch.empty(rows, K, dtype=torch.bfloat16, device=like.device)
    if sync is None:
        sync = torch.empty(4, dtype=torch.int32, device=like.device)
    return xn, sync


def norm_linear_bf16(a, gamma, eps: float, b, c, xn=None, sync=None, stream=None) -> torch.Tensor:
    """c = RMSNorm(a) b^T, the norm in the GEMM's prologue (c bf16 or fp32); returns xn, the
    normalised rows the GEMM multiplied (into `xn` if given)."""
    M, K = a.shape
    xn, sync = _norm_buffers(M, K, a, xn, sync)
    N.check(N.lib().llama_norm_linear_bf16(_ptr(a), _ptr(gamma), eps, _ptr(b), _ptr(c), M, b.shape[0], K,
                                           int(c.dtype == torch.float32), _ptr(xn), _ptr(sync), _stream(stream)),
            "llama_norm_linear_bf16")
    return xn


def norm_linear_swiglu(a, gamma, eps: float, w_gate, w_up, out, xn=None, sync=None, stream=None) -> torch.Tensor:
    M, K = a.shape
    xn, sync = _norm_buffers(M, K, a, xn, sync)
    N.check(N.lib().llama_norm_linear_swiglu(_ptr(a), _ptr(gamma), eps, _ptr(w_gate), _ptr(w_up), _ptr(out), M,
                                             w_gate.shape[0], K, _ptr(xn), _ptr(sync), _stream(stream)),
            "llama_norm_linear_swiglu")
    return xn


def norm_qkv_rope(dims: Dims, x, attn_norm, wq, wk, wv, cos, sin, cache_k, cache_v, q_out, xn=None, sync=None,
                  stream=None) -> torch.Tensor:
    B, S = x.shape[0], x.shape[1]
    xn, sync = _norm_buffers(B * S, x.shape[-1], x, xn, sync)
    d = dims.c()
    N.check(N.lib().llama_norm_qkv_rope(ctypes.byref(d), _ptr(x), _ptr(attn_norm), _ptr(wq), _ptr(wk), _ptr(wv),
                                        _ptr(cos), _ptr(sin), cos.shape[0], cache_struct(cache_k, cache_v),
                                        _ptr(q_out), B, S, _ptr(xn), _ptr(sync), _stream(stream)),
            "llama_norm_qkv_rope")
    return xn


def prefill_intermediates(dims: Dims, ws, B: int, S: int, offset: int = 0) -> dict:
    """Views of the workspace regions where the last llama_layer_prefill(_chunk) call on `ws`
    (its layer workspace starting `offset` bytes in) left q [B, H, S, D], the attention output
    o [B, S, H*D], h [B, S, d], the gated MLP activation a [B, S, d_inter] and hn =
    RMSNorm_2(h) [B, S, d].  Read them after that call has completed on its stream."""
    offs = (ctypes.c_size_t * 5)()
    d = dims.c()
    N.check(N.lib().llama_layer_prefill_workspace_layout(ctypes.byref(d), B, S, offs), "workspace layout")
    es = 2 if dims.dtype == torch.bfloat16 else 4
    shapes = {"q": (B, dims.n_heads, S, dims.head_dim), "o": (B, S, dims.n_heads * dims.head_dim),
              "h": (B, S, dims.d_model), "a": (B, S, dims.d_inter), "hn": (B, S, dims.d_model)}
    out = {}
    for off, (name, shape) in zip(offs, shapes.items()):
        n = int(np.prod(shape))
        out[name] = ws[offset + off:offset + off + n * es].view(dims.dtype).view(shape)
    return out


def stack_intermediates(st: "StackArgs", ws, B: int, S: int) -> dict:
    """After llama_stack_forward on `ws`: its last layer's input x and output, plus that layer's
    intermediates (prefill_intermediates)."""
    offs = (ctypes.c_size_t * 3)()
    N.check(N.lib().llama_stack_workspace_layout(ctypes.byref(st.s), B, S, offs), "stack workspace layout")
    dims = st.dims
    es = 2 if dims.dtype == torch.bfloat16 else 4
    n = B * S * dims.d_model * es
    out = prefill_intermediates(dims, ws, B, S, offs[2])
    out["x"] = ws[offs[0]:offs[0] + n].view(dims.dtype).view(B, S, dims.d_model)
    out["out"] = ws[offs[1]:offs[1] + n].view(dims.dtype).view(B, S, dims.d_model)
    return out


def attention_prefill(dims: Dims, q, cache_k, cache_v, out, stream=None) -> None:
    B, _, S, _ = q.shape
    d = dims.c()
    N.check(N.lib().llama_attention_prefill(ctypes.byref(d), _ptr(q), cache_struct(cache_k, cache_v), _ptr(out), B, S,
                                            _stream(stream)), "llama_attention_prefill")


def attention_decode_workspace_bytes(dims: Dims, B: int, max_T: int) -> int:
    n = ctypes.c_size_t()
    d = dims.c()
    N.check(N.lib().llama_attention_decode_workspace_bytes(ctypes.byref(d), B, max_T, ctypes.byref(n)), "workspace")
    return n.value


def attention_decode(dims: Dims, q, cache_k, cache_v, positions, out, ws, stream=None) -> None:
    d = dims.c()
    N.check(N.lib().llama_attention_decode(ctypes.byref(d), _ptr(q), cache_struct(cache_k, cache_v), _ptr(positions),
                                           _ptr(out), q.shape[0], _ptr(ws), ws.numel(), _stream(stream)),
            "llama_attention_decode")


def device_status(stream=None) -> int:
    """Synchronises the stream; returns and clears the device status word."""
    return N.lib().llama_get_device_status(_stream(stream))


def wait_probe(budget_ns: int, stream=None) -> None:
    N.check(N.lib().llama_debug_wait_probe(budget_ns, _stream(stream)), "llama_debug_wait_probe")


def timeout_record() -> dict:
    """Where the first timed-out device wait gave up (all zeros if none did)."""
    buf = (ctypes.c_int64 * 7)()
    N.check(N.lib().llama_debug_timeout_record(buf, 7), "llama_debug_timeout_record")
    r = list(buf)
    return {"waited_ns": r[0], "polls": r[1], "block": (r[2] & 0xffffffff, r[2] >> 32), "thread": r[3],
            "sm": r[4], "barrier_smem": r[5] & 0xffffffff, "parity": r[5] >> 32,
            "grid": (r[6] & 0xffffffff, r[6] >> 32)}


def launch_count() -> int:
    return N.lib().llama_kernel_launch_count()


class KernelTrace:
    """Times every kernel that the library enqueues inside a ``with`` block (CUDA events
    recorded by the library on its launch stream after each kernel)."""

    def __init__(self, max_kernels: int = 64, stream=None):
        self.stream = stream or torch.cuda.current_stream()
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(max_kernels + 1)]
        for e in self.events:           # torch creates the CUDA event on first record
            e.record(self.stream)
        self.handles = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self.n = 0

    def __enter__(self):
        N.check(N.lib().llama_trace_begin(self.handles, len(self.events), self.stream.cuda_stream), "trace_begin")
        return self

    def __exit__(self, *exc):
        self.n = N.lib().llama_trace_end()
        return False

    def kernel_ms(self) -> list[float]:
        """Duration of each traced kernel, after the stream has been synchronised."""
        return [self.events[i].elapsed_time(self.events[i + 1]) for i in range(self.n - 1)]
