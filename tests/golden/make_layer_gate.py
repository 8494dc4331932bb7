"""Derives the full-width whole-layer gate (tests/golden/layer_gate.json) from the oracle alone.

The GPU tests compare the whole bf16 layer at d = 4096 with the oracle run from x: the MHA-7B
layer on all 2048 rows, and the GQA-8B layer on the first 256 rows of each of its 4 sequences
(an exact causal prefix).  There a correct implementation cannot meet 2e-2 * (1 + |ref|) at
every element (tests/numerics_model.py explains why), so those two comparisons use a gate
derived here, before and without any GPU result:

  1. the exact oracle on exactly those rows;
  2. the oracle with the numerics of this library's kernels -- fp32 accumulation noise before
     every bf16 storage rounding and bf16 softmax probabilities in the attention -- for five
     noise seeds; the RMSNorm rounding point needs no term (the norm-fused GEMMs round where the
     oracle does);
  3. each effect alone at seed 0, to show where the deviation comes from;
  4. the gate: over both workloads and all seeds, 1.5 x the largest elementwise maximum and
     normwise distance, and 2 x the largest fraction of elements above 2e-2 (a GPU run is one
     more draw from the same distribution; the margins cover draws beyond five seeds).

Run from the repository root: python tests/golden/make_layer_gate.py  (a few minutes, CPU)
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path[:0] = [ROOT, os.path.join(ROOT, "tests")]

import oracle  # noqa: E402
import numerics_model as nm  # noqa: E402
from llama_decoder_block_gb300 import synth  # noqa: E402

CASES = {"mha7b_bf16_b1_s2048": 2048, "gqa8b_bf16_b4_s4096": 256}   # workload -> rows per sequence checked
SEEDS = range(5)
GPU_EFFECTS = ("noise", "p_bf16")
TOL = 2e-2


def case_inputs(name, rows):
    wl = synth.WORKLOADS[name]
    L = wl.layer
    w = {k: v.f64() for k, v in synth.layer_weights(wl).items()}
    x = synth.activations(wl).f64()[:, :rows]
    c, s = oracle.rope_tables(L.rope_base, L.head_dim, rows)
    c, s = c.astype(np.float32).astype(np.float64), s.astype(np.float32).astype(np.float64)
    kw = dict(n_heads=L.n_heads, n_kv_heads=L.n_kv_heads, head_dim=L.head_dim, rms_eps=L.rms_eps, store_bf16=True)
    return x, w, c, s, kw


def model_deviation(name, rows, effects, seed, ref=None):
    x, w, c, s, kw = case_inputs(name, rows)
    if ref is None:
        ref, _, _ = oracle.decoder_layer(x, w, c, s, **kw)
    with nm.model_numerics(effects, seed=seed):
        out, _, _ = oracle.decoder_layer(x, w, c, s, **kw)
    return nm.deviation(out, ref, TOL), ref


def derive():
    result = {"tol": TOL, "effects": list(GPU_EFFECTS), "cases": {}}
    for name, rows in CASES.items():
        x, w, c, s, kw = case_inputs(name, rows)
        ref, _, _ = oracle.decoder_layer(x, w, c, s, **kw)
        case = {"rows_per_sequence": rows, "seeds": {}, "alone_seed0": {}}
        for seed in SEEDS:
            with nm.model_numerics(GPU_EFFECTS, seed=seed):
                out, _, _ = oracle.decoder_layer(x, w, c, s, **kw)
            case["seeds"][str(seed)] = nm.deviation(out, ref, TOL)
            print(name, "seed", seed, case["seeds"][str(seed)], flush=True)
        for eff in GPU_EFFECTS:
            with nm.model_numerics((eff,), seed=0):
                out, _, _ = oracle.decoder_layer(x, w, c, s, **kw)
            case["alone_seed0"][eff] = nm.deviation(out, ref, TOL)
            print(name, eff, "alone", case["alone_seed0"][eff], flush=True)
        result["cases"][name] = case
    result["gate"] = gate_from(result)
    return result


def gate_from(result):
    runs = [d for case in result["cases"].values() for d in case["seeds"].values()]
    return {"tol": result["tol"],
            "envelope": round(1.5 * max(d["max"] for d in runs), 4),
            "normwise": round(1.5 * max(d["normwise"] for d in runs), 5),
            "max_frac_over_tol": round(2.0 * max(d["frac_over_tol"] for d in runs), 6)}


if __name__ == "__main__":
    res = derive()
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "layer_gate.json")
    with open(path, "w", encoding="utf-8") as f:
        json.dump(res, f, indent=1)
        f.write("\n")
    print(json.dumps(res["gate"]))
