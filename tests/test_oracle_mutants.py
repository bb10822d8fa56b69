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


# ----------------------------------------------------- the numpy-level oracle
# Planted mistakes in the functions written in Python (packed sequences, the
# dt transform, the gate, bf16 rounding): each mutant replaces one oracle
# function for the duration of a pin test, which must then fail.
import tests.test_oracle_pins as pins

_scan_varlen, _dt_transform, _gate, _round_bf16, _step = (
    oracle.scan_varlen, oracle.dt_transform, oracle.gate, oracle.round_bf16, oracle.step)


def _varlen_shared_init(x, dt, A, B, C, cu, D=None, init=None, nthreads=None):
    shared = None if init is None else np.repeat(np.asarray(init)[:1], len(cu) - 1, axis=0)
    return _scan_varlen(x, dt, A, B, C, cu, D, shared, nthreads)


def _varlen_state_carried(x, dt, A, B, C, cu, D=None, init=None, nthreads=None):
    y = np.empty(np.shape(x), np.float64)
    fin = np.zeros((len(cu) - 1,) + np.shape(x)[1:] + (np.shape(B)[2],), np.float64)
    h = None if init is None else np.asarray(init, np.float64)[:1]
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if a < b:
            ys, h = oracle.scan_seq(x[None, a:b], dt[None, a:b], A, B[None, a:b], C[None, a:b], D, h)
            y[a:b] = ys[0]
        fin[s] = 0 if h is None else h[0]
    return y, fin


def _varlen_offset_shift(x, dt, A, B, C, cu, D=None, init=None, nthreads=None):
    cu2 = np.asarray(cu).copy()
    cu2[1:-1] += 1
    return _scan_varlen(x, dt, A, B, C, cu2, D, init, nthreads)


def _gate_sigmoid_only(y, z):
    z = np.asarray(z, np.float64)
    return np.asarray(y, np.float64) * np.exp(-np.logaddexp(0.0, -z))


def _gate_wrong_sign(y, z):
    z = np.asarray(z, np.float64)
    return np.asarray(y, np.float64) * (z * np.exp(-np.logaddexp(0.0, z)))


def _round_half_up(a):
    m, e = np.frexp(np.asarray(a, np.float64))
    return np.ldexp(np.floor(m * 256.0 + 0.5) / 256.0, e)


def _round_truncate(a):
    m, e = np.frexp(np.asarray(a, np.float64))
    return np.ldexp(np.trunc(m * 256.0) / 256.0, e)


def _dt_bias_after_softplus(dt, bias=None, softplus=False, lo=-np.inf, hi=np.inf):
    u = np.asarray(dt, np.float64)
    if softplus:
        u = np.logaddexp(0.0, u)
    if bias is not None:
        u = u + np.asarray(bias, np.float64)
    return np.minimum(np.maximum(u, lo), hi)


def _dt_clamp_first(dt, bias=None, softplus=False, lo=-np.inf, hi=np.inf):
    u = np.asarray(dt, np.float64)
    if bias is not None:
        u = u + np.asarray(bias, np.float64)
    u = np.minimum(np.maximum(u, lo), hi)
    return np.logaddexp(0.0, u) if softplus else u


def _bf16_step_rounds_y(state, x, dt, A, B, C, D=None, nthreads=None):
    y, st = _step(state, x, dt, A, B, C, D, nthreads)
    return _round_bf16(y), _round_bf16(st)


def _bf16_step_unrounded(state, x, dt, A, B, C, D=None, nthreads=None):
    return _step(state, x, dt, A, B, C, D, nthreads)


def _rel_over_result(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    den = float(np.linalg.norm(got.ravel()))
    num = float(np.linalg.norm((got - ref).ravel()))
    return num / den if den > 0 else num


def _rel_squared(got, ref):
    return _REL(got, ref) ** 2


def _rel_max_norm(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    den = float(np.max(np.abs(ref)))
    num = float(np.max(np.abs(got - ref)))
    return num / den if den > 0 else num


def _rel_matrix_norm(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if got.ndim != 2:
        return _REL(got, ref)
    den = float(np.linalg.norm(ref, 2))
    num = float(np.linalg.norm(got - ref, 2))
    return num / den if den > 0 else num


def _rel_zero_ref_divides(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        return float(np.float64(np.linalg.norm((got - ref).ravel()))
                     / np.float64(np.linalg.norm(ref.ravel())))


def _e4m3_parts(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(c >> 7, -1.0, 1.0), (c >> 3) & 15, (c & 7).astype(np.float64), c


def _e4m3_bias_8(codes):
    sign, e, m, c = _e4m3_parts(codes)
    mag = np.where(e == 0, np.ldexp(m, -10), np.ldexp(1.0 + m / 8.0, e - 8))
    return sign * np.where((c & 0x7F) == 0x7F, np.nan, mag)


def _e4m3_no_subnormals(codes):
    sign, e, m, c = _e4m3_parts(codes)
    mag = np.ldexp(1.0 + m / 8.0, e - 7)
    return sign * np.where((c & 0x7F) == 0x7F, np.nan, mag)


def _e4m3_subnormal_scale_2m10(codes):
    sign, e, m, c = _e4m3_parts(codes)
    mag = np.where(e == 0, np.ldexp(m, -10), np.ldexp(1.0 + m / 8.0, e - 7))
    return sign * np.where((c & 0x7F) == 0x7F, np.nan, mag)


def _e4m3_with_infinities(codes):
    sign, e, m, c = _e4m3_parts(codes)
    mag = np.where(e == 0, np.ldexp(m, -9), np.ldexp(1.0 + m / 8.0, e - 7))
    return sign * np.where(e == 15, np.where(m == 0, np.inf, np.nan), mag)


def _e4m3_unsigned(codes):
    sign, e, m, c = _e4m3_parts(codes)
    mag = np.where(e == 0, np.ldexp(m, -9), np.ldexp(1.0 + m / 8.0, e - 7))
    return np.where((c & 0x7F) == 0x7F, np.nan, mag)


_REL = oracle.rel_l2

PY_MUTANTS = {
    "varlen_shared_initial_state": ("scan_varlen", _varlen_shared_init,
                                    pins.test_varlen_is_each_sequence_alone_by_quadratic_form),
    "varlen_state_leaks_across_sequences": ("scan_varlen", _varlen_state_carried,
                                            pins.test_varlen_is_each_sequence_alone_by_quadratic_form),
    "varlen_offsets_shifted": ("scan_varlen", _varlen_offset_shift,
                               pins.test_varlen_is_each_sequence_alone_by_quadratic_form),
    "gate_sigmoid_without_z": ("gate", _gate_sigmoid_only, pins.test_gate_closed_forms),
    "gate_sigmoid_of_minus_z": ("gate", _gate_wrong_sign, pins.test_gate_closed_forms),
    "bf16_ties_away_from_zero": ("round_bf16", _round_half_up, pins.test_round_bf16_nearest_even),
    "bf16_truncation": ("round_bf16", _round_truncate, pins.test_round_bf16_nearest_even),
    "dt_bias_after_softplus": ("dt_transform", _dt_bias_after_softplus,
                               pins.test_dt_transform_bias_per_head_then_clamp),
    "dt_clamp_before_softplus": ("dt_transform", _dt_clamp_first,
                                 pins.test_dt_transform_bias_per_head_then_clamp),
    "bf16_step_rounds_y": ("step_bf16_state", _bf16_step_rounds_y,
                           pins.test_step_bf16_state_is_rounded_step),
    "bf16_step_state_not_rounded": ("step_bf16_state", _bf16_step_unrounded,
                                    pins.test_step_bf16_state_is_rounded_step),
    "rel_l2_divided_by_result_norm": ("rel_l2", _rel_over_result,
                                      pins.test_rel_l2_on_hand_worked_values),
    "rel_l2_squared": ("rel_l2", _rel_squared, pins.test_rel_l2_on_hand_worked_values),
    "rel_l2_max_norm": ("rel_l2", _rel_max_norm, pins.test_rel_l2_on_hand_worked_values),
    "rel_l2_matrix_norm": ("rel_l2", _rel_matrix_norm, pins.test_rel_l2_on_hand_worked_values),
    "rel_l2_zero_reference_divides": ("rel_l2", _rel_zero_ref_divides,
                                      pins.test_rel_l2_on_hand_worked_values),
    "e4m3_exponent_bias_8": ("decode_e4m3", _e4m3_bias_8, pins.test_decode_e4m3_closed_forms),
    "e4m3_subnormals_as_normals": ("decode_e4m3", _e4m3_no_subnormals,
                                   pins.test_decode_e4m3_closed_forms),
    "e4m3_subnormal_scale": ("decode_e4m3", _e4m3_subnormal_scale_2m10,
                             pins.test_decode_e4m3_closed_forms),
    "e4m3_top_exponent_reserved": ("decode_e4m3", _e4m3_with_infinities,
                                   pins.test_decode_e4m3_closed_forms),
    "e4m3_sign_dropped": ("decode_e4m3", _e4m3_unsigned, pins.test_decode_e4m3_closed_forms),
    "e4m3_bias_8_against_torch": ("decode_e4m3", _e4m3_bias_8,
                                  pins.test_decode_e4m3_equals_torch_float8_for_every_code),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_pins_catch_planted_python_mistake(name, monkeypatch):
    attr, mutant, pin = PY_MUTANTS[name]
    monkeypatch.setattr(oracle, attr, mutant)
    with pytest.raises(AssertionError):
        pin()
