"""Plants plausible mistakes in a copy of the oracle (on the CPU) and checks that the pins catch each one."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "eps_outside_sqrt": ("return gamma * (x * (1.0 / np.sqrt(ms + eps)))", "return gamma * (x / (np.sqrt(ms) + eps))"),
    "norm_subtracts_mean": ("ms = np.mean(x * x, axis=-1, keepdims=True)",
                            "x = x - x.mean(-1, keepdims=True); ms = np.mean(x * x, axis=-1, keepdims=True)"),
    "layernorm_unbiased_variance": ("var = np.mean((x - mu) ** 2, axis=-1, keepdims=True)",
                                    "var = np.sum((x - mu) ** 2, axis=-1, keepdims=True) / (x.shape[-1] - 1)"),
    "layernorm_eps_outside_sqrt": ("return gamma * ((x - mu) / np.sqrt(var + eps)) + beta",
                                   "return gamma * ((x - mu) / (np.sqrt(var) + eps)) + beta"),
    "layernorm_beta_scaled": ("return gamma * ((x - mu) / np.sqrt(var + eps)) + beta",
                              "return gamma * ((x - mu) / np.sqrt(var + eps) + beta)"),
    "rope_half_split": ("x_even = x[..., 0::2]\n    x_odd = x[..., 1::2]",
                        "x_even = x[..., :x.shape[-1]//2]\n    x_odd = x[..., x.shape[-1]//2:]"),
    "rope_half_interleaved": ("    x1 = x[..., :half]\n    x2 = x[..., half:]", "    x1 = x[..., 0::2]\n    x2 = x[..., 1::2]"),
    "rope_half_sign": ("y[..., half:] = x2 * cos + x1 * sin", "y[..., half:] = x2 * cos - x1 * sin"),
    "rope_sign": ("y[..., 0::2] = x_even * cos - x_odd * sin", "y[..., 0::2] = x_even * cos + x_odd * sin"),
    "rope_frequency": ("theta = np.power(float(base), -2.0 * i / head_dim)", "theta = np.power(float(base), -1.0 * i / head_dim)"),
    "rope_on_v": ("    v = st(v)\n", "    v = st(apply_rope(v, c, s))\n"),
    "group_map_modulo": ("g = h // rep", "g = h % G"),
    "mask_strict": ("allowed = np.arange(T)[None, :] <= np.asarray(q_pos[b])[:, None]",
                    "allowed = np.arange(T)[None, :] < np.maximum(np.asarray(q_pos[b])[:, None], 1)"),
    "scale_1_over_D": ("scores = (q[b, h] @ k[b, g, :T].T) / np.sqrt(D)", "scores = (q[b, h] @ k[b, g, :T].T) / D"),
    "silu_on_up": ("return store(silu(x @ w_gate.T) * (x @ w_up.T)) @ w_down.T",
                   "return store(silu(x @ w_up.T) * (x @ w_gate.T)) @ w_down.T"),
    "bf16_truncates": ("return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)", "return np.ldexp(np.trunc(np.ldexp(m, 8)), e - 8)"),
    "residual_after_norm": ("    residual = x\n    xn = st(rms_norm(x, w[\"attn_norm\"], rms_eps))",
                            "    xn = st(rms_norm(x, w[\"attn_norm\"], rms_eps))\n    residual = xn"),
    "shared_norm_gamma": ("hn = st(rms_norm(h, w[\"ffn_norm\"], rms_eps))",
                          "hn = st(rms_norm(h, w[\"attn_norm\"], rms_eps))"),
    "no_final_norm": ("xn = rms_norm(x, final_norm, rms_eps)", "xn = x"),
    "stack_decode_no_final_norm": ("xn = rms_norm(x[:, 0], final_norm, rms_eps)", "xn = x[:, 0]"),
    "stack_decode_cache_of_wrong_layer": ("for w, (pk, pv) in zip(layers, caches):",
                                          "for w, (pk, pv) in zip(layers, caches[::-1]):"),
    "decode_positions_restart": ("pos = past_len[:, None] + np.arange(S)[None, :]",
                                 "pos = np.zeros_like(past_len)[:, None] + np.arange(S)[None, :]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "layer.py"), encoding="utf-8").read()
    assert before in src
    for d in ("oracle", "tests", "llama_decoder_block_gb300"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d,
                        ignore=shutil.ignore_patterns("__pycache__", "*.so", "csrc"))
    (tmp_path / "oracle" / "layer.py").write_text(src.replace(before, after), encoding="utf-8")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
