"""ctypes declarations of the C ABI in include/llama_layer.h (argument marshalling only).

Loading fails with an exception when libllama_layer.so is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libllama_layer.so")

c_int32, c_float, c_void_p, c_size_t = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
c_double, c_uint64 = ctypes.c_double, ctypes.c_uint64

LLAMA_F32, LLAMA_BF16 = 0, 1
STATUS = {0: "LLAMA_OK", -1: "LLAMA_ERR_INVALID_ARG", -2: "LLAMA_ERR_UNSUPPORTED", -3: "LLAMA_ERR_CUDA",
          -4: "LLAMA_ERR_TIMEOUT", -5: "LLAMA_ERR_DEVICE_BOUNDS", -6: "LLAMA_ERR_SCRATCH_LIMIT"}


class LayerDims(ctypes.Structure):
    _fields_ = [("d_model", c_int32), ("n_heads", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32),
                ("d_inter", c_int32), ("rms_eps", c_float), ("dtype", c_int32), ("rope_style", c_int32)]


WEIGHT_FIELDS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in WEIGHT_FIELDS]


class KVCache(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("max_T", c_int32)]


class Stack(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("vocab", c_int32), ("dims", LayerDims),
                ("layers", ctypes.POINTER(LayerWeights)), ("final_norm", c_void_p), ("embed", c_void_p),
                ("lm_head", c_void_p)]


P = ctypes.POINTER
# name -> (restype, argtypes), one entry per declaration in include/llama_layer.h
SIGNATURES = {
    "llama_layer_prefill_workspace_bytes": (c_int32, [P(LayerDims), c_int32, c_int32, P(c_size_t)]),
    "llama_layer_prefill": (c_int32, [P(LayerDims), P(LayerWeights), c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_int32, KVCache, c_int32, c_int32, c_void_p, c_size_t, c_void_p]),
    "llama_layer_prefill_chunk": (c_int32, [P(LayerDims), P(LayerWeights), c_void_p, c_void_p, c_void_p, c_void_p,
                                            c_int32, c_void_p, c_void_p, KVCache, c_int32, c_int32, c_void_p,
                                            c_size_t, c_void_p]),
    "llama_layer_decode_workspace_bytes": (c_int32, [P(LayerDims), c_int32, c_int32, P(c_size_t)]),
    "llama_layer_decode": (c_int32, [P(LayerDims), P(LayerWeights), c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                     c_void_p, KVCache, c_int32, c_void_p, c_size_t, c_void_p]),
    "llama_stack_workspace_bytes": (c_int32, [P(Stack), c_int32, c_int32, P(c_size_t)]),
    "llama_stack_forward": (c_int32, [P(Stack), c_void_p, c_void_p, c_void_p, c_void_p, c_int32, P(KVCache),
                                      c_int32, c_int32, c_void_p, c_size_t, c_void_p]),
    "llama_stack_decode_workspace_bytes": (c_int32, [P(Stack), c_int32, P(c_size_t)]),
    "llama_stack_decode": (c_int32, [P(Stack), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                     P(KVCache), c_int32, c_void_p, c_size_t, c_void_p]),
    "llama_stack_decode_graph": (c_int32, [P(Stack), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                           P(KVCache), c_int32, c_void_p, c_size_t, P(c_void_p)]),
    "llama_graph_launch": (c_int32, [c_void_p, c_void_p]),
    "llama_graph_kernel_count": (c_int32, [c_void_p]),
    "llama_graph_destroy": (c_int32, [c_void_p]),
    "llama_rmsnorm": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_float, c_int32, c_void_p]),
    "llama_layernorm": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_float, c_int32,
                                  c_void_p]),
    "llama_linear_bf16": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p]),
    "llama_linear_residual": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                        c_void_p]),
    "llama_linear_swiglu": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p]),
    "llama_qkv_rope": (c_int32, [P(LayerDims), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                 KVCache, c_void_p, c_int32, c_int32, c_void_p]),
    "llama_norm_linear_bf16": (c_int32, [c_void_p, c_void_p, c_float, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                         c_int32, c_void_p, c_void_p, c_void_p]),
    "llama_norm_linear_swiglu": (c_int32, [c_void_p, c_void_p, c_float, c_void_p, c_void_p, c_void_p, c_int32,
                                           c_int32, c_int32, c_void_p, c_void_p, c_void_p]),
    "llama_norm_qkv_rope": (c_int32, [P(LayerDims), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_int32, KVCache, c_void_p, c_int32, c_int32, c_void_p, c_void_p,
                                      c_void_p]),
    "llama_layer_prefill_workspace_layout": (c_int32, [P(LayerDims), c_int32, c_int32, P(c_size_t)]),
    "llama_stack_workspace_layout": (c_int32, [P(Stack), c_int32, c_int32, P(c_size_t)]),
    "llama_attention_prefill": (c_int32, [P(LayerDims), c_void_p, KVCache, c_void_p, c_int32, c_int32, c_void_p]),
    "llama_attention_decode_workspace_bytes": (c_int32, [P(LayerDims), c_int32, c_int32, P(c_size_t)]),
    "llama_attention_decode": (c_int32, [P(LayerDims), c_void_p, KVCache, c_void_p, c_void_p, c_int32, c_void_p,
                                         c_size_t, c_void_p]),
    "llama_attention_decode_static": (c_int32, [P(LayerDims), c_void_p, KVCache, c_void_p, c_void_p, c_int32,
                                                c_void_p]),
    "llama_rope_tables": (c_int32, [c_double, c_int32, c_int32, c_void_p, c_void_p]),
    "llama_get_device_status": (c_int32, [c_void_p]),
    "llama_status_string": (ctypes.c_char_p, [c_int32]),
    "llama_debug_wait_probe": (c_int32, [c_uint64, c_void_p]),
    "llama_debug_timeout_record": (c_int32, [ctypes.POINTER(ctypes.c_int64), c_int32]),
    "llama_kernel_launch_count": (c_uint64, []),
    "llama_trace_begin": (c_int32, [ctypes.POINTER(c_void_p), c_int32, c_void_p]),
    "llama_trace_end": (c_int32, []),
}

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                        "(there is no fallback implementation)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


class LlamaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({lib().llama_status_string(code).decode()})")


def check(code: int, where: str) -> None:
    if code != 0:
        raise LlamaError(code, where)
