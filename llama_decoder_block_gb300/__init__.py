"""GB300 (sm_103a) LLaMA-style pre-norm decoder layer: hand-written CUDA behind a C ABI.

``api`` is the Python binding of ``include/llama_layer.h``; ``synth`` draws the seeded
synthetic inputs; ``build`` compiles ``libllama_layer.so`` in-tree.
"""
