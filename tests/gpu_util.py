"""Helpers of the GPU parity tests: moving synth tensors to the device and the tolerance check."""
import contextlib

import numpy as np
import torch

from llama_decoder_block_gb300 import api, synth

# |gpu - ref| <= TOL * (1 + |ref|), elementwise
TOL = {"f32": 1e-4, "bf16": 2e-2}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}
NAN_BF16 = np.uint16(0x7FC0)


def to_dev(s: synth.Stored, device="cuda") -> torch.Tensor:
    if s.dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(s.data).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(s.data)).to(device)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_stored(a: np.ndarray) -> synth.Stored:
    return synth.Stored(synth.f32_to_bf16_bits(a.astype(np.float32)), "bf16")


# Every comparison made by the helpers below: (what, max, p99 of |gpu-ref|/(1+|ref|), gate).
# tests/conftest.py writes them out at the end of the session when LLAMA_PARITY_LOG names a file.
PARITY_LOG = []


def assert_close(gpu: np.ndarray, ref: np.ndarray, tol: float, what: str):
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values in the GPU result"
    err = np.abs(gpu - ref) / (1.0 + np.abs(ref))
    PARITY_LOG.append((what, float(err.max()), float(np.quantile(err, 0.99)), f"max <= {tol:.0e}"))
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, (f"{what}: max |gpu-ref|/(1+|ref|) = {err.max():.3e} > {tol:.0e} at {worst} "
                              f"(gpu {gpu[worst]!r}, ref {ref[worst]!r}); p99 {np.quantile(err, 0.99):.3e}")
    return float(err.max())


# Whole bf16 layer at full width (d = 4096, d_inter = 11008 / 14336): bf16 storage of the
# activations makes two correct implementations differ by more than TOL at a few elements.
# The oracle itself, computed the way a tensor-core implementation does (fp32-sized noise,
# 2e-7 relative, before each bf16 storage rounding; softmax probabilities rounded to bf16
# before they multiply V), moves at the GQA 8B shape by up to 4.3e-2, with 1.2e-3 of the
# elements above 2e-2 and 3.2e-3 normwise (tests/test_oracle_sensitivity.py).  Gate: TOL on
# all but 3e-3 of the elements, ENVELOPE everywhere, NORMWISE on the whole tensor.
LAYER_FULL = {"tol": 2e-2, "max_frac_over_tol": 3e-3, "envelope": 6e-2, "normwise": 5e-3}


def assert_close_layer_full(gpu: np.ndarray, ref: np.ndarray, what: str):
    g = LAYER_FULL
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values in the GPU result"
    err = np.abs(gpu - ref) / (1.0 + np.abs(ref))
    frac = float(np.mean(err > g["tol"]))
    norm = float(np.linalg.norm(gpu - ref) / np.linalg.norm(ref))
    PARITY_LOG.append((what, float(err.max()), float(np.quantile(err, 0.99)),
                       f"full-width gate: frac over {g['tol']:.0e} = {frac:.2e}, normwise {norm:.2e}"))
    msg = (f"{what}: max {err.max():.3e} (envelope {g['envelope']:.0e}), fraction over {g['tol']:.0e} = {frac:.2e} "
           f"(limit {g['max_frac_over_tol']:.0e}), normwise {norm:.2e} (limit {g['normwise']:.0e}), "
           f"p99 {np.quantile(err, 0.99):.2e}")
    assert err.max() <= g["envelope"] and frac <= g["max_frac_over_tol"] and norm <= g["normwise"], msg
    return msg


def attention_bf16_probabilities(q, k, v, q_pos, k_len):
    """The oracle's attention with the probabilities rounded to bf16 before the product with
    V and the normaliser summed from the unrounded ones (flash-attention numerics)."""
    import oracle
    B, H, S, D = q.shape
    rep = H // k.shape[1]
    out = np.empty_like(q)
    for b in range(B):
        T = int(k_len[b])
        allowed = np.arange(T)[None, :] <= np.asarray(q_pos[b])[:, None]
        for h in range(H):
            g = h // rep
            scores = np.where(allowed, (q[b, h] @ k[b, g, :T].T) / np.sqrt(D), -np.inf)
            p = np.exp(scores - scores.max(axis=-1, keepdims=True))
            out[b, h] = (oracle.round_bf16(p) @ v[b, g, :T]) / p.sum(axis=-1, keepdims=True)
    return out


@contextlib.contextmanager
def tensor_core_numerics(seed=0):
    """Within the block the oracle computes the way a tensor-core implementation does:
    fp32-sized relative noise (2e-7) before each bf16 storage rounding, and bf16 softmax
    probabilities.  Comparing it with the exact oracle measures how far a correct bf16
    implementation lands from the oracle for a given workload."""
    from oracle import layer as oracle_layer
    exact_round, exact_attention = oracle_layer.round_bf16, oracle_layer.attention
    rng = np.random.default_rng(seed)
    oracle_layer.round_bf16 = lambda v: exact_round(np.asarray(v, np.float64) *
                                                    (1 + 2e-7 * rng.standard_normal(np.shape(v))))
    oracle_layer.attention = attention_bf16_probabilities
    try:
        yield
    finally:
        oracle_layer.round_bf16, oracle_layer.attention = exact_round, exact_attention


def deviation(a: np.ndarray, ref: np.ndarray) -> dict:
    err = np.abs(a - ref) / (1.0 + np.abs(ref))
    return {"max": float(err.max()), "p99": float(np.quantile(err, 0.99)),
            "normwise": float(np.linalg.norm(a - ref) / np.linalg.norm(ref))}


def gen_layer(args):
    """Process-pool worker: one layer's weights of a workload (storage format)."""
    wl, layer = args
    return synth.layer_weights(wl, layer)


def dims_of(layer: synth.LayerShape) -> api.Dims:
    return api.Dims(layer.d_model, layer.n_heads, layer.n_kv_heads, layer.head_dim, layer.d_inter, layer.rms_eps,
                    TORCH_DT[layer.dtype], {"even_odd": 0, "half": 1}[layer.rope_style])


def tables(layer: synth.LayerShape, max_pos: int, oracle_mod, device="cuda"):
    """RoPE tables made by the oracle in fp64 and rounded to fp32: the same input on both sides."""
    c, s = oracle_mod.rope_tables(layer.rope_base, layer.head_dim, max_pos)
    c32, s32 = c.astype(np.float32), s.astype(np.float32)
    return (torch.from_numpy(c32).to(device), torch.from_numpy(s32).to(device),
            c32.astype(np.float64), s32.astype(np.float64))


def oracle_kw(layer: synth.LayerShape) -> dict:
    return dict(n_heads=layer.n_heads, n_kv_heads=layer.n_kv_heads, head_dim=layer.head_dim, rms_eps=layer.rms_eps,
                rope=layer.rope_style)
