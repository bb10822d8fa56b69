"""Pins for the fp64 oracle: each test checks it against something other than
itself -- the quadratic (dual) form, closed forms, a hand-derived example,
invariances the mathematics fixes.

The recurrence being pinned is the Mamba-2 state update of the CGLA kernel
page ("Mamba-Family State-Space Model Kernels on a Programmable CGLA",
section III.A): h_t = exp(dt_t A) h_{t-1} + dt_t B_t x_t^T,
y_t = C_t . h_t + D x_t, with diagonal per-head dynamics ("Compiler-First
State Space Duality ...", abstract).  The pages print no SSD values, so no pin
is a value taken from them.
"""
import json
import os

import numpy as np
import pytest

import oracle
from state_space_model_chunked_gb300 import inputs as gen

HERE = os.path.dirname(os.path.abspath(__file__))


def _quadratic(x, dt, A, B, C, D, init):
    """The dual (masked, attention-like) form of the scan, written from the
    unrolled recurrence: y_t = sum_{s<=t} (C_t.B_s) exp(cum_t - cum_s) dt_s x_s
    + exp(cum_t) C_t.h0 + D x_t, cum = inclusive cumsum of dt*A."""
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros((b, L, H, P))
    fin = np.zeros((b, H, P, N))
    t_idx = np.arange(L)
    causal = t_idx[:, None] >= t_idx[None, :]
    for bi in range(b):
        for h in range(H):
            g = h // (H // G)
            cum = np.cumsum(dt[bi, :, h].astype(np.float64) * float(A[h]))
            diff = np.where(causal, cum[:, None] - cum[None, :], -np.inf)
            Lmask = np.exp(diff)
            Cg = C[bi, :, g, :].astype(np.float64)
            Bg = B[bi, :, g, :].astype(np.float64)
            X = x[bi, :, h, :].astype(np.float64)
            M = (Cg @ Bg.T) * Lmask * dt[bi, :, h].astype(np.float64)[None, :]
            yy = M @ X
            if init is not None:
                h0 = init[bi, h].astype(np.float64)          # [P][N]
                yy += np.exp(cum)[:, None] * (Cg @ h0.T)
            if D is not None:
                yy += float(D[h]) * X
            y[bi, :, h, :] = yy
            w = np.exp(cum[-1] - cum) * dt[bi, :, h]
            f = (X * w[:, None]).T @ Bg                       # [P][N]
            if init is not None:
                f += np.exp(cum[-1]) * init[bi, h].astype(np.float64)
            fin[bi, h] = f
    return y, fin


def _rel(a, b):
    return oracle.rel_l2(a, b)


@pytest.mark.parametrize("H,G,P,N,L", [(1, 1, 4, 5, 37), (3, 1, 5, 4, 64),
                                        (3, 3, 4, 4, 50), (4, 2, 5, 4, 41)])
@pytest.mark.parametrize("with_init", [False, True])
def test_seq_matches_quadratic_form(H, G, P, N, L, with_init):
    inp = gen.scan_inputs(2, L, H, P, N, G, "f32", seed=11 + H + L,
                          random_init=with_init)
    y, fin = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init"], nthreads=2)
    yq, fq = _quadratic(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                        inp["D"], inp["init"])
    assert _rel(y, yq) < 1e-10
    assert _rel(fin, fq) < 1e-10


def test_hand_worked_example():
    g = json.load(open(os.path.join(HERE, "golden", "hand_example_L3.json")))
    i = g["inputs"]
    x = np.array(i["x"]).reshape(1, 3, 1, 1)
    dt = np.array(i["dt"]).reshape(1, 3, 1)
    A = np.array(i["A"])
    B = np.array(i["B"]).reshape(1, 3, 1, 2)
    C = np.array(i["C"]).reshape(1, 3, 1, 2)
    D = np.array(i["D"])
    init = np.array(i["init"]).reshape(1, 1, 1, 2)
    y, fin = oracle.scan_seq(x, dt, A, B, C, D, init)
    tol = g["tolerance"]
    np.testing.assert_allclose(y.ravel(), g["expected"]["y"], rtol=tol, atol=tol)
    np.testing.assert_allclose(fin.ravel(), np.ravel(g["expected"]["final_state"]),
                               rtol=tol, atol=tol)


def test_A_zero_is_prefix_sum():
    inp = gen.scan_inputs(1, 40, 2, 3, 4, 1, "f32", seed=3, random_init=True)
    A = np.zeros(2)
    y, fin = oracle.scan_seq(inp["x"], inp["dt"], A, inp["B"], inp["C"], None,
                             inp["init"])
    x, dt, B, C, h0 = (inp[k].astype(np.float64) for k in ("x", "dt", "B", "C", "init"))
    for h in range(2):
        # outer products dt_s x_s B_s^T, accumulated
        terms = dt[0, :, h, None, None] * x[0, :, h, :, None] * B[0, :, 0, None, :]
        hs = h0[0, h][None] + np.cumsum(terms, axis=0)          # [L][P][N]
        ys = np.einsum("tpn,tn->tp", hs, C[0, :, 0, :])
        assert _rel(y[0, :, h], ys) < 1e-12
        assert _rel(fin[0, h], hs[-1]) < 1e-12


def test_constant_decay_is_geometric_series():
    L, P, N = 30, 3, 4
    rng = np.random.default_rng(5)
    alpha_dt, A = 0.05, -2.0            # dt*A = -0.1 for every token
    x1 = rng.standard_normal(P)
    B1 = rng.standard_normal(N)
    C1 = rng.standard_normal(N)
    h0 = rng.standard_normal((P, N))
    x = np.tile(x1, (1, L, 1, 1)).reshape(1, L, 1, P)
    dt = np.full((1, L, 1), alpha_dt)
    B = np.tile(B1, (1, L, 1, 1)).reshape(1, L, 1, N)
    C = np.tile(C1, (1, L, 1, 1)).reshape(1, L, 1, N)
    y, fin = oracle.scan_seq(x, dt, np.array([A]), B, C, np.array([0.7]),
                             h0.reshape(1, 1, P, N))
    a = alpha_dt * A
    for t in range(L):
        k = t + 1
        ht = np.exp(a * k) * h0 + alpha_dt * np.outer(x1, B1) * (1 - np.exp(a * k)) / (1 - np.exp(a))
        np.testing.assert_allclose(y[0, t, 0], ht @ C1 + 0.7 * x1, rtol=1e-12, atol=1e-12)
    hL = np.exp(a * L) * h0 + alpha_dt * np.outer(x1, B1) * (1 - np.exp(a * L)) / (1 - np.exp(a))
    np.testing.assert_allclose(fin[0, 0], hL, rtol=1e-12, atol=1e-12)


def test_zero_input_is_pure_decay():
    inp = gen.scan_inputs(2, 33, 3, 4, 5, 1, "f32", seed=9, random_init=True)
    x = np.zeros_like(inp["x"])
    y, fin = oracle.scan_seq(x, inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["init"])
    for b in range(2):
        for h in range(3):
            cum = np.cumsum(inp["dt"][b, :, h].astype(np.float64) * float(inp["A"][h]))
            h0 = inp["init"][b, h].astype(np.float64)
            ys = np.exp(cum)[:, None] * (inp["C"][b, :, 0, :].astype(np.float64) @ h0.T)
            assert _rel(y[b, :, h], ys) < 1e-12
            assert _rel(fin[b, h], np.exp(cum[-1]) * h0) < 1e-12


@pytest.mark.parametrize("Q", [16, 32, 64, 256, 48])
def test_chunk_size_invariance(Q):
    inp = gen.scan_inputs(2, 200, 3, 8, 16, 1, "bf16", seed=21, random_init=True)
    ys, fs = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init"])
    yc, fc, S, Hp = oracle.scan_chunked(inp["x"], inp["dt"], inp["A"], inp["B"],
                                        inp["C"], Q, inp["D"], inp["init"],
                                        want_intermediates=True)
    assert _rel(yc, ys) < 1e-12
    assert _rel(fc, fs) < 1e-12
    # exposed intermediates obey the inter-chunk recurrence
    nc = S.shape[1]
    assert _rel(Hp[:, 0], inp["init"]) < 1e-15
    for c in range(nc - 1):
        lo, hi = c * Q, min((c + 1) * Q, 200)
        dec = np.exp(np.sum(inp["dt"][:, lo:hi, :].astype(np.float64) * inp["A"][None, None, :], axis=1))
        nxt = dec[:, :, None, None] * Hp[:, c] + S[:, c]
        assert _rel(Hp[:, c + 1], nxt) < 1e-12


def test_chunk_intermediates_are_their_definition():
    # S_c of one chunk equals the final state of that chunk scanned alone
    # from a zero state (the definition of a chunk's own contribution).
    inp = gen.scan_inputs(1, 96, 2, 4, 8, 1, "f32", seed=4)
    Q = 32
    _, _, S, Hp = oracle.scan_chunked(inp["x"], inp["dt"], inp["A"], inp["B"],
                                      inp["C"], Q, inp["D"], None,
                                      want_intermediates=True)
    for c in range(3):
        sl = slice(c * Q, (c + 1) * Q)
        _, fq = _quadratic(inp["x"][:, sl], inp["dt"][:, sl], inp["A"],
                           inp["B"][:, sl], inp["C"][:, sl], None, None)
        assert _rel(S[:, c], fq) < 1e-12


@pytest.mark.parametrize("k", [1, 57, 128])
def test_split_resume_invariance(k):
    inp = gen.scan_inputs(2, 160, 2, 6, 8, 1, "bf16", seed=31, random_init=True)
    y, fin = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init"])
    a = {kk: (v[:, :k] if kk in ("x", "dt", "B", "C") else v) for kk, v in inp.items()}
    b = {kk: (v[:, k:] if kk in ("x", "dt", "B", "C") else v) for kk, v in inp.items()}
    y1, f1 = oracle.scan_seq(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["init"])
    y2, f2 = oracle.scan_seq(b["x"], b["dt"], b["A"], b["B"], b["C"], b["D"], f1)
    assert _rel(np.concatenate([y1, y2], axis=1), y) < 1e-13
    assert _rel(f2, fin) < 1e-13


def test_prefill_equals_decode_steps():
    inp = gen.scan_inputs(2, 24, 4, 4, 8, 2, "bf16", seed=41, random_init=True)
    y, fin = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init"])
    st = inp["init"].astype(np.float64)
    for t in range(24):
        yt, st = oracle.step(st, inp["x"][:, t], inp["dt"][:, t], inp["A"],
                             inp["B"][:, t], inp["C"][:, t], inp["D"])
        assert _rel(yt, y[:, t]) < 1e-13
    assert _rel(st, fin) < 1e-13


def test_linearity_in_x_and_init():
    i1 = gen.scan_inputs(1, 50, 2, 4, 6, 1, "f32", seed=51, random_init=True)
    i2 = gen.scan_inputs(1, 50, 2, 4, 6, 1, "f32", seed=52, random_init=True)
    al, be = 0.75, -1.25
    common = dict(dt=i1["dt"], A=i1["A"], B=i1["B"], C=i1["C"], D=i1["D"])
    y1, f1 = oracle.scan_seq(i1["x"], init=i1["init"], **common)
    y2, f2 = oracle.scan_seq(i2["x"], init=i2["init"], **common)
    x1, x2 = i1["x"].astype(np.float64), i2["x"].astype(np.float64)
    h1, h2 = i1["init"].astype(np.float64), i2["init"].astype(np.float64)
    y3, f3 = oracle.scan_seq(al * x1 + be * x2, init=al * h1 + be * h2,
                             **common)
    assert _rel(y3, al * y1 + be * y2) < 1e-13
    assert _rel(f3, al * f1 + be * f2) < 1e-13


def test_thread_count_does_not_change_result():
    inp = gen.scan_inputs(3, 70, 5, 4, 8, 1, "bf16", seed=61, random_init=True)
    y1, f1 = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init"], nthreads=1)
    y4, f4 = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                             inp["D"], inp["init"], nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(f1, f4)


def test_bf16_rounding_is_nearest_even():
    # values chosen at and around bf16 rounding boundaries
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 2**-8 + 2**-20, 1.0 + 3 * 2**-8,
                     -2.5, 3.0e-3], np.float32)
    got, bits = gen.bf16_round(vals)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa -> 1.0
    # 1 + 3*2^-8 is a tie between 1+2^-7 and 1+2^-6 ... even -> 1 + 2^-6
    assert got[0] == 1.0
    assert got[1] == 1.0
    assert got[2] == np.float32(1.0 + 2**-7)
    assert got[3] == np.float32(1.0 + 2**-6)
    assert got[4] == -2.5
    assert abs(got[5] - 3.0e-3) <= 3.0e-3 * 2**-8
    assert bits[0] == 0x3F80


# ------------------------------------------------------------- dt transform
def test_dt_transform_identity_by_default():
    dt = np.random.default_rng(1).uniform(-3, 3, size=(2, 5, 3)).astype(np.float32)
    out = oracle.dt_transform(dt)
    assert out.dtype == np.float64 and np.array_equal(out, dt.astype(np.float64))


def test_dt_transform_softplus_closed_forms():
    """softplus(0) = ln 2; for large u, softplus(u) = u + log1p(e^-u); for very
    negative u, softplus(u) = e^u (1 - e^u/2 + ...)."""
    assert oracle.dt_transform(np.zeros(1), softplus=True)[0] == np.log(2.0)
    u = np.array([30.0, 50.0, 800.0])
    assert np.allclose(oracle.dt_transform(u, softplus=True), u + np.log1p(np.exp(-u)),
                       rtol=0, atol=1e-12)
    v = np.array([-30.0, -50.0])
    assert np.allclose(oracle.dt_transform(v, softplus=True), np.exp(v), rtol=1e-12)
    w = np.linspace(-5, 5, 101)
    assert np.allclose(oracle.dt_transform(w, softplus=True), np.log(1.0 + np.exp(w)),
                       rtol=1e-14)


def test_dt_transform_bias_per_head_then_clamp():
    dt = np.zeros((1, 4, 3))
    bias = np.array([-1.0, 0.5, 3.0])
    out = oracle.dt_transform(dt, bias)
    assert np.array_equal(out, np.broadcast_to(bias, (1, 4, 3)))
    out = oracle.dt_transform(dt, bias, lo=0.0, hi=1.0)
    assert np.array_equal(out[0, 0], [0.0, 0.5, 1.0])
    # softplus of the biased value, then the clamp (order matters)
    out = oracle.dt_transform(dt, bias, softplus=True, lo=0.5, hi=2.0)
    assert np.allclose(out[0, 0], [0.5, np.log1p(np.exp(0.5)), 2.0], rtol=1e-15)



# ---------------------------------------------------------------- packed sequences
def test_varlen_is_each_sequence_alone_by_quadratic_form():
    """Packed sequences: every sequence is its own scan from its own initial
    state (the per-sequence recurrence of CGLA section III.A); checked per
    sequence against the dual form, so state leaking across a boundary, a
    shifted offset or a shared initial state fails.  An empty sequence keeps
    its initial state."""
    lengths = [5, 0, 13, 1, 9]
    inp = gen.varlen_inputs(lengths, 3, 4, 8, 1, "bf16", seed=77, random_init=True)
    y, fin = oracle.scan_varlen(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                inp["cu"], inp["D"], inp["init"])
    cu = inp["cu"]
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        if a == b:
            np.testing.assert_array_equal(fin[s], inp["init"][s])
            continue
        yq, fq = _quadratic(inp["x"][None, a:b], inp["dt"][None, a:b], inp["A"],
                            inp["B"][None, a:b], inp["C"][None, a:b], inp["D"],
                            inp["init"][s:s + 1])
        assert _rel(y[a:b], yq[0]) < 1e-12
        assert _rel(fin[s], fq[0]) < 1e-12


def test_varlen_equal_lengths_is_the_batched_scan():
    """Sequences of one length packed end to end are the batched layout with
    the batch axis flattened into the token axis."""
    b, L = 3, 17
    inp = gen.scan_inputs(b, L, 2, 4, 8, 2, "f32", seed=5, random_init=True)
    cu = np.arange(b + 1) * L
    y, fin = oracle.scan_varlen(inp["x"].reshape(b * L, 2, 4), inp["dt"].reshape(b * L, 2),
                                inp["A"], inp["B"].reshape(b * L, 2, 8),
                                inp["C"].reshape(b * L, 2, 8), cu, inp["D"], inp["init"])
    yb, fb = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["init"])
    np.testing.assert_array_equal(y, yb.reshape(b * L, 2, 4))
    np.testing.assert_array_equal(fin, fb)


def test_varlen_empty_sequence_without_init_is_zero_state():
    inp = gen.varlen_inputs([0, 4], 2, 4, 8, 1, "f32", seed=3)
    _, fin = oracle.scan_varlen(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                inp["cu"], inp["D"])
    assert not fin[0].any() and fin[1].any()


# ---------------------------------------------------------------- output gate
def test_gate_closed_forms():
    """silu(0) = 0; silu(1) = 1 / (1 + e^-1); silu(z) - silu(-z) = z (the
    sigmoid's halves sum to one); silu(z) -> z for large z and -> 0 for very
    negative z; the gate is y times that, per element."""
    y = np.array([2.0, -3.0, 0.5, 1.0, 1.0])
    z = np.array([0.0, 1.0, 40.0, -40.0, -800.0])
    g = oracle.gate(y, z)
    assert g[0] == 0.0
    assert abs(g[1] - (-3.0) / (1.0 + np.exp(-1.0))) < 1e-15
    assert abs(g[2] - 0.5 * 40.0) < 1e-12
    assert abs(g[3]) < 1e-15 and g[4] == 0.0 and np.isfinite(g).all()
    w = np.linspace(-6, 6, 97)
    ones = np.ones_like(w)
    assert np.allclose(oracle.gate(ones, w) - oracle.gate(ones, -w), w, rtol=0, atol=1e-14)


# ---------------------------------------------------------------- bf16 states
def test_round_bf16_nearest_even():
    """bf16 keeps 8 significant bits: at 1 the spacing is 2^-7, ties go to the
    even significand, exactly representable values stay, signs are symmetric,
    and the rounding agrees with the bit-level encoder of the input module."""
    u = 2.0 ** -7
    vals = np.array([1.0, 1 + u / 2, 1 + 1.5 * u, 1 + u / 2 + 2.0 ** -20, -(1 + 1.5 * u), 3.0,
                     0.1])
    want = np.array([1.0, 1.0, 1 + 2 * u, 1 + u, -(1 + 2 * u), 3.0, 0.10009765625])
    np.testing.assert_array_equal(oracle.round_bf16(vals), want)
    r = np.random.default_rng(4).standard_normal(10000).astype(np.float32)
    np.testing.assert_array_equal(oracle.round_bf16(r), gen.bf16_round(r)[0].astype(np.float64))


def test_step_bf16_state_is_rounded_step():
    """The bf16-state step: y from the unrounded fp64 update, the state that
    update rounded; with A = 0, dt = 1 and x = 0 the state is unchanged and
    already bf16, so rounding is the identity."""
    b, H, P, N, G = 2, 3, 4, 8, 1
    st = gen.bf16_round(gen.decode_state(b, H, P, N, seed=2))[0]
    tok = gen.decode_token_inputs(b, H, P, N, G, "bf16", seed=2)
    A = np.full(H, -0.5, np.float32)
    y, s = oracle.step_bf16_state(st, tok["x"], tok["dt"], A, tok["B"], tok["C"])
    y0, s0 = oracle.step(st, tok["x"], tok["dt"], A, tok["B"], tok["C"])
    np.testing.assert_array_equal(y, y0)
    np.testing.assert_array_equal(s, oracle.round_bf16(s0))
    assert np.abs(s - s0).max() <= np.abs(s0).max() * 2.0 ** -8
    y1, s1 = oracle.step_bf16_state(st, np.zeros_like(tok["x"]), np.ones_like(tok["dt"]),
                                    np.zeros(H, np.float32), tok["B"], tok["C"])
    np.testing.assert_array_equal(s1, st.astype(np.float64))


def test_hand_worked_packed_example():
    """Packed sequences against values worked out by hand (including an empty
    sequence whose state must come back unchanged)."""
    g = json.load(open(os.path.join(HERE, "golden", "hand_example_packed.json")))
    i = g["inputs"]
    T = len(i["x"])
    y, fin = oracle.scan_varlen(np.array(i["x"]).reshape(T, 1, 1), np.array(i["dt"]).reshape(T, 1),
                                np.array(i["A"]), np.array(i["B"]).reshape(T, 1, 1),
                                np.array(i["C"]).reshape(T, 1, 1), np.array(i["cu"]),
                                np.array(i["D"]), np.array(i["init"]).reshape(3, 1, 1, 1))
    tol = g["tolerance"]
    np.testing.assert_allclose(y.ravel(), g["expected"]["y"], rtol=tol, atol=tol)
    np.testing.assert_allclose(fin.ravel(), g["expected"]["final_state"], rtol=tol, atol=tol)


def test_rel_l2_on_hand_worked_values():
    """The parity measure itself (relative L2 over the whole tensor, reading
    c11), on values worked out by hand.  Each case separates it from a
    plausible slip: dividing by the norm of the result under test, squaring
    the ratio, a max-norm or L1 norm, a per-element mean, a matrix (spectral)
    norm of a 2-D array, and a division by a zero reference."""
    # ||(0,0) - (3,4)|| / ||(3,4)|| = 5 / 5
    assert oracle.rel_l2([0.0, 0.0], [3.0, 4.0]) == 1.0
    # half the reference: ||(1.5,2)|| / ||(3,4)|| = 2.5 / 5
    assert oracle.rel_l2([1.5, 2.0], [3.0, 4.0]) == 0.5
    # error (0,1) against (3,4): 1/5 (max-norm 1/4, L1 1/7, squared 1/25)
    assert abs(oracle.rel_l2([3.0, 5.0], [3.0, 4.0]) - 0.2) < 1e-15
    # twice the reference: the error norm equals the reference norm (dividing
    # by the result's norm would give 1/2)
    assert oracle.rel_l2([6.0, 8.0], [3.0, 4.0]) == 1.0
    # 2-D: error all ones (Frobenius 2) against 3 I (Frobenius 3 sqrt 2) ->
    # sqrt(2)/3; the spectral norms would give 2/3
    ref = 3.0 * np.eye(2)
    assert abs(oracle.rel_l2(ref + 1.0, ref) - np.sqrt(2.0) / 3.0) < 1e-15
    # an all-zero reference: the absolute norm, ||(1,2,2)|| = 3
    assert oracle.rel_l2([1.0, 2.0, 2.0], [0.0, 0.0, 0.0]) == 3.0
    # the same elements in another order and shape give the same value
    a = np.arange(12.0).reshape(3, 4)
    b = a + np.linspace(-1.0, 1.0, 12).reshape(3, 4)
    perm = np.random.default_rng(0).permutation(12)
    assert oracle.rel_l2(b, a) == pytest.approx(oracle.rel_l2(b.ravel()[perm], a.ravel()[perm]),
                                                rel=1e-15)


# ---------------------------------------------------------------- fp8 (E4M3) decode
def test_decode_e4m3_equals_torch_float8_for_every_code():
    """All 256 codes against torch's float8_e4m3fn -> float64 conversion (a
    library routine independent of the oracle): equal values, NaN at the
    same two codes."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_decode_e4m3_closed_forms():
    """Values the encoding's definition fixes: the subnormals step by 2^-9 up to
    7 * 2^-9 and meet the smallest normal 2^-6 one step later; 0x38 is
    exponent field 7 (= the bias) with a zero significand, i.e. 1; the
    largest finite value (1 + 6/8) 2^8 = 448 sits just below the NaN code; the
    sign bit only negates."""
    d = oracle.decode_e4m3
    assert d(np.uint8(0x00)) == 0.0 and np.signbit(d(np.uint8(0x80)))
    sub = d(np.arange(0, 8, dtype=np.uint8))
    np.testing.assert_array_equal(sub, np.arange(8) * 2.0 ** -9)
    assert d(np.uint8(0x08)) == 2.0 ** -6 == d(np.uint8(0x07)) + 2.0 ** -9
    assert d(np.uint8(0x38)) == 1.0
    assert d(np.uint8(0x3C)) == 1.5 and d(np.uint8(0x40)) == 2.0
    assert d(np.uint8(0x7E)) == 448.0
    assert np.isnan(d(np.uint8(0x7F))) and np.isnan(d(np.uint8(0xFF)))
    pos = d(np.arange(0x00, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)                       # strictly increasing
    neg = d(np.arange(0x80, 0xFF, dtype=np.uint8))
    np.testing.assert_array_equal(neg, -pos)


def test_every_e4m3_value_is_a_bfloat16_value():
    """The fp8 path widens E4M3 to bfloat16 and relies on that being exact:
    every finite E4M3 value survives rounding to bfloat16 unchanged."""
    v = oracle.decode_e4m3(np.arange(256, dtype=np.uint8))
    v = v[np.isfinite(v) & (v != 0)]
    np.testing.assert_array_equal(oracle.round_bf16(v), v)


def test_fp8_inputs_decode_to_the_drawn_distribution():
    """The seeded fp8 inputs are codes of N(0, 1) draws: decoded, they match
    the bf16-rounded draws of the same seed within E4M3's half spacing (2^-4
    relative; 2^-10 absolute for subnormals) plus bfloat16's (2^-9)."""
    a = gen.scan_inputs(1, 300, 4, 32, 16, 1, "fp8", seed=5)
    b = gen.scan_inputs(1, 300, 4, 32, 16, 1, "bf16", seed=5)
    for k in ("x", "B", "C"):
        assert a[k].dtype == np.uint8
        v = oracle.decode_e4m3(a[k])
        assert np.all(np.isfinite(v))
        err = np.abs(v - b[k])
        bound = np.maximum(np.abs(b[k]) * (2.0 ** -4 + 2.0 ** -8), 2.0 ** -10 + 2.0 ** -16)
        assert np.all(err <= bound), k
    np.testing.assert_array_equal(a["dt"], b["dt"])
