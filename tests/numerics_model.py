"""A model of how far a correct bf16 tensor-core implementation of the layer lands from the oracle.

The oracle (oracle/layer.py) computes each step exactly in fp64 and rounds to bf16 only where
the configurations store an activation.  A GPU implementation differs from it in three ways,
each harmless on its own but amplified by every later bf16 storage rounding (a value near a
rounding boundary lands on the neighbouring bf16 number, and the flip moves everything
downstream of it; the d_inter-long down projection sums those moves):

  noise   fp32 accumulation: the value before each storage rounding carries a relative error
          of about 1e-7 (modelled as 2e-7 * N(0, 1));
  p_bf16  attention with tensor cores multiplies V by the softmax probabilities rounded to bf16
          (the normaliser is summed from the unrounded ones);
  norm    the RMSNorm-fused GEMMs round the normalised operand as bf16(gamma * x) and apply the
          row factor rsqrt(mean(x^2) + eps) to the fp32 product, not before the rounding.

``model_numerics`` switches any subset of them on inside the oracle (test infrastructure only:
it patches the oracle module's own functions for the duration of a ``with`` block).
"""
from __future__ import annotations

import contextlib

import numpy as np

from oracle import layer as oracle_layer

EFFECTS = ("noise", "p_bf16", "norm")


def attention_bf16_probabilities(q, k, v, q_pos, k_len):
    """The oracle's attention with the probabilities rounded to bf16 before the product with V
    and the normaliser summed from the unrounded ones (flash-attention numerics)."""
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
            out[b, h] = (oracle_layer.round_bf16(p) @ v[b, g, :T]) / p.sum(axis=-1, keepdims=True)
    return out


@contextlib.contextmanager
def model_numerics(effects=EFFECTS, seed=0):
    """Inside the block the oracle computes with the chosen effects (a subset of EFFECTS)."""
    effects = set(effects)
    assert effects <= set(EFFECTS), effects
    exact_round, exact_attention, exact_norm = oracle_layer.round_bf16, oracle_layer.attention, oracle_layer.rms_norm
    rng = np.random.default_rng(seed)
    passed = []   # the fused norm's output: the storage rounding that follows leaves it as it is

    def rounding(v):
        if passed and v is passed[-1]:
            return passed.pop()
        v = np.asarray(v, np.float64)
        if "noise" in effects:
            v = v * (1 + 2e-7 * rng.standard_normal(np.shape(v)))
        return exact_round(v)

    def fused_norm(x, gamma, eps):
        # gamma * x of two bf16 numbers is exact in fp32, so only its bf16 rounding is modelled
        r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
        passed[:] = [exact_round(gamma * x) * r]
        return passed[0]

    oracle_layer.round_bf16 = rounding
    if "p_bf16" in effects:
        oracle_layer.attention = attention_bf16_probabilities
    if "norm" in effects:
        oracle_layer.rms_norm = fused_norm
    try:
        yield
    finally:
        oracle_layer.round_bf16, oracle_layer.attention, oracle_layer.rms_norm = exact_round, exact_attention, exact_norm


def deviation(a: np.ndarray, ref: np.ndarray, tol: float = 2e-2) -> dict:
    """max and p99 of |a - ref| / (1 + |ref|), the fraction above `tol`, and the normwise distance."""
    err = np.abs(a - ref) / (1.0 + np.abs(ref))
    return {"max": float(err.max()), "p99": float(np.quantile(err, 0.99)), "frac_over_tol": float(np.mean(err > tol)),
            "normwise": float(np.linalg.norm(a - ref) / np.linalg.norm(ref))}
