"""CPU oracle of the LLaMA-style pre-norm decoder layer -- TEST INFRASTRUCTURE ONLY.

Plain fp64 numpy, written from the pages' definitions, sharing no code with the
CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference arm may import it; the product path never does.
"""
from .layer import (  # noqa: F401
    round_bf16, linear, rms_norm, layer_norm, rope_tables, apply_rope, apply_rope_half, silu, swiglu_mlp,
    attention, decoder_layer, stack_forward, stack_decode, param_count, kv_cache_bytes,
)
