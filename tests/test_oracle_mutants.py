"""Planted mistakes: each test copies the oracle's C source, plants one
plausible error in the sequential recurrence (on the CPU, in a temporary
build), and checks that the pins catch it.  This is evidence that the pins in
test_oracle_pins.py constrain every term of the recurrence."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from state_space_model_chunked_gb300 import inputs as gen
from tests.test_oracle_pins import _quadratic

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

MUTANTS = {
    "output_uses_state_before_update": (
        "row[n] = abar * row[n] + dx * Bt[n];\n                acc += Ct[n] * row[n];",
        "acc += Ct[n] * row[n];\n                row[n] = abar * row[n] + dx * Bt[n];"),
    "skip_scaled_by_dt": ("yt[p] = acc + Dh * xt[p];", "yt[p] = acc + Dh * dx;"),
    "groups_interleaved": ("const int64_t g = h / (H / G);", "const int64_t g = h % G;"),
    "decay_without_dt": ("exp(dtv * j->A[h])", "exp(j->A[h])"),
    "input_not_dt_scaled": ("const double dx = dtv * xt[p];", "const double dx = xt[p];"),
    "readout_with_B": ("acc += Ct[n] * row[n];", "acc += Bt[n] * row[n];"),
    "init_batch_head_swapped": ("j->init + (b * H + h) * P * N", "j->init + (h * j->batch + b) * P * N"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    str(c), "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    ref = oracle._load()
    lib.oracle_scan_seq.restype = ref.oracle_scan_seq.restype
    lib.oracle_scan_seq.argtypes = ref.oracle_scan_seq.argtypes
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name, monkeypatch):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    inp = gen.scan_inputs(2, 41, 4, 5, 4, 2, "f32", seed=77, random_init=True)
    yq, fq = _quadratic(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                        inp["D"], inp["init"])
    monkeypatch.setattr(oracle, "_lib", lib)
    y, fin = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init"])
    caught = oracle.rel_l2(y, yq) > 1e-6 or oracle.rel_l2(fin, fq) > 1e-6
    assert caught, f"pin did not catch mutant {name}"


def test_unmutated_source_passes(tmp_path, monkeypatch):
    lib = _build_mutant(tmp_path, "none", "exp(", "exp(")
    inp = gen.scan_inputs(2, 41, 4, 5, 4, 2, "f32", seed=77, random_init=True)
    yq, fq = _quadratic(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                        inp["D"], inp["init"])
    monkeypatch.setattr(oracle, "_lib", lib)
    y, fin = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init"])
    assert oracle.rel_l2(y, yq) < 1e-10 and oracle.rel_l2(fin, fq) < 1e-10
    assert np.isfinite(y).all()
