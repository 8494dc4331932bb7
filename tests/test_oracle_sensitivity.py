"""The full-width whole-layer gate (tests/golden/layer_gate.json) and the derivation behind it.

tests/golden/make_layer_gate.py computes, from the oracle alone, how far the oracle with this
library's kernel numerics (fp32 noise before each bf16 storage rounding, bf16 softmax
probabilities; tests/numerics_model.py) lands from the exact oracle, for five noise seeds, on
exactly the rows the GPU's full-width tests check, and sets the gate from those runs.  These
tests re-run one of the stored cases and check that the stored gate follows from the stored
runs by the stated rule, and that the plain elementwise band is too tight for any of them.
"""
import json
import os

import numpy as np
import pytest

import numerics_model as nm
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(HERE, "golden", "layer_gate.json"), encoding="utf-8") as _f:
    GATE = json.load(_f)


def _derivation():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_layer_gate", os.path.join(HERE, "golden", "make_layer_gate.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_stored_gate_follows_from_the_stored_runs():
    mod = _derivation()
    assert GATE["gate"] == mod.gate_from(GATE)
    assert set(GATE["cases"]) == set(mod.CASES) and GATE["effects"] == list(mod.GPU_EFFECTS)
    for case in GATE["cases"].values():
        assert len(case["seeds"]) == len(mod.SEEDS)
        for d in case["seeds"].values():
            # a correct bf16 implementation already leaves the plain band at some elements
            assert d["max"] > GATE["tol"]
            assert d["max"] <= GATE["gate"]["envelope"] and d["normwise"] <= GATE["gate"]["normwise"]
            assert d["frac_over_tol"] <= GATE["gate"]["max_frac_over_tol"]


def test_one_stored_run_reproduces():
    # the GQA-8B case (first 256 rows of 4 sequences) at seed 0: the same numbers again
    mod = _derivation()
    name = "gqa8b_bf16_b4_s4096"
    got, _ = mod.model_deviation(name, mod.CASES[name], mod.GPU_EFFECTS, seed=0)
    want = GATE["cases"][name]["seeds"]["0"]
    for k in ("max", "p99", "frac_over_tol", "normwise"):
        assert got[k] == pytest.approx(want[k], rel=1e-9), k


def test_model_numerics_switch_off_cleanly():
    # outside the block the oracle is itself again
    x = np.array([[3.0, 4.0]])
    before = oracle.rms_norm(x, np.ones(2), 0.0)
    with nm.model_numerics(nm.EFFECTS, seed=1):
        pass
    assert np.array_equal(oracle.rms_norm(x, np.ones(2), 0.0), before)
    assert oracle.round_bf16(1.0 + 2.0 ** -9) == 1.0      # ties to even, unpatched
