"""Helpers of the GPU parity tests: moving synth tensors to the device and the tolerance check."""
import json
import os

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
# activations makes two correct implementations differ by more than TOL at a few elements
# (tests/numerics_model.py).  The gate comes from tests/golden/layer_gate.json, which
# tests/golden/make_layer_gate.py derives from the oracle alone: the oracle computed with this
# library's kernel numerics, five noise seeds, on exactly the rows the full-width tests check.
# Gate: TOL on all but `max_frac_over_tol` of the elements, `envelope` everywhere, `normwise`
# on the whole tensor.  Each step of the layer is held to TOL itself (test_gpu_teacher_forced.py).
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "layer_gate.json"),
          encoding="utf-8") as _f:
    LAYER_FULL = json.load(_f)["gate"]


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


def deviation(a: np.ndarray, ref: np.ndarray) -> dict:
    err = np.abs(a - ref) / (1.0 + np.abs(ref))
    return {"max": float(err.max()), "p99": float(np.quantile(err, 0.99)),
            "frac_over_tol": float(np.mean(err > TOL["bf16"])),
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
