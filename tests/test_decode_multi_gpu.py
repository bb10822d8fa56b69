"""GPU parity of the multi-token decode (ssd_state_update_multi): T tokens per
(batch, head) in one call, the state read and written once, against T
chained fp64 oracle steps, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_chunked_gb300 import inputs as gen
from tests.gpu_util import TOL, dev, host, rel

pytestmark = pytest.mark.gpu


def _tokens(b, T, H, P, N, G, dtype, seed):
    """T per-token decode inputs stacked on a token axis: x [b,T,H,P],
    dt [b,T,H], B/C [b,T,G,N]."""
    toks = [gen.decode_token_inputs(b, H, P, N, G, dtype, seed=seed, step=t) for t in range(T)]
    return {k: np.stack([t[k] for t in toks], axis=1) for k in ("x", "dt", "B", "C")}


def _oracle_steps(state, tok, A, D, dt_kw=None, z=None):
    """T chained oracle.step calls; returns (y [b,T,H,P], final state)."""
    s = state.astype(np.float64)
    ys = []
    for t in range(tok["x"].shape[1]):
        dt = tok["dt"][:, t]
        if dt_kw:
            dt = oracle.dt_transform(dt, **dt_kw)
        y, s = oracle.step(s, tok["x"][:, t], dt, A, tok["B"][:, t], tok["C"][:, t], D)
        if z is not None:
            y = oracle.gate(y, z[:, t])
        ys.append(y)
    return np.stack(ys, axis=1), s


@pytest.mark.parametrize("T", [1, 4, 16, 37])
@pytest.mark.parametrize("b,H,P,N,G", [
    (2, 80, 64, 128, 1),        # one 2.7B-shaped layer
    (3, 6, 20, 32, 2),          # ragged headdim, two groups
    (1, 4, 64, 256, 2),         # widest state
    (2, 3, 7, 4, 1),            # narrowest state, odd headdim
    (1, 2, 200, 16, 1),         # long rows of a narrow state
    (2, 5, 24, 8, 1),           # two float4 per row, one thread per row
    (2, 4, 128, 64, 2),         # the widest headdim of a 64-wide state
])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_multi_token_decode_matches_chained_steps(T, b, H, P, N, G, dtype):
    import state_space_model_chunked_gb300 as ssd
    seed = 11 * T + N + P
    state = gen.decode_state(b, H, P, N, seed=seed)
    A, D = gen.decode_params(H, seed=seed)
    tok = _tokens(b, T, H, P, N, G, dtype, seed)
    s_dev = dev(state)
    y = ssd.state_update_multi(s_dev, dev(tok["x"], dtype), dev(tok["dt"]), dev(A),
                               dev(tok["B"], dtype), dev(tok["C"], dtype), dev(D))
    torch.cuda.synchronize()
    y_ref, s_ref = _oracle_steps(state, tok, A, D)
    assert rel(host(y), y_ref) <= TOL[dtype], rel(host(y), y_ref)
    # the update itself is fp32 arithmetic on exact inputs
    assert rel(host(s_dev), s_ref) <= 1e-5, rel(host(s_dev), s_ref)
    ssd.last_device_error()


def test_multi_token_decode_equals_single_token_calls():
    """The same 16 tokens through 16 ssd_state_update calls: the states agree
    to fp32 rounding (the multi-token kernel carries a scaled state, so the
    roundings differ)."""
    import state_space_model_chunked_gb300 as ssd
    b, T, H, P, N, G = 2, 16, 8, 64, 128, 2
    state = gen.decode_state(b, H, P, N, seed=5)
    A, D = gen.decode_params(H, seed=5)
    tok = _tokens(b, T, H, P, N, G, "bf16", 5)
    s_multi, s_single = dev(state), dev(state)
    y_multi = ssd.state_update_multi(s_multi, dev(tok["x"], "bf16"), dev(tok["dt"]), dev(A),
                                     dev(tok["B"], "bf16"), dev(tok["C"], "bf16"), dev(D))
    ys = []
    for t in range(T):
        ys.append(ssd.state_update(s_single, dev(tok["x"][:, t], "bf16"), dev(tok["dt"][:, t]),
                                   dev(A), dev(tok["B"][:, t], "bf16"),
                                   dev(tok["C"][:, t], "bf16"), dev(D)))
    torch.cuda.synchronize()
    assert rel(host(s_multi), host(s_single)) <= 1e-6
    assert rel(host(y_multi), host(torch.stack(ys, dim=1))) <= 1e-2


def test_multi_token_decode_bf16_state_rounded_once():
    """A bf16 state: fp32 updates over all tokens, rounded to bf16 once at the
    write-back; y from the unrounded updates."""
    import state_space_model_chunked_gb300 as ssd
    b, T, H, P, N, G = 2, 8, 16, 64, 128, 1
    state = oracle.round_bf16(gen.decode_state(b, H, P, N, seed=9)).astype(np.float32)
    A, D = gen.decode_params(H, seed=9)
    tok = _tokens(b, T, H, P, N, G, "bf16", 9)
    s_dev = dev(state, "bf16")
    y = ssd.state_update_multi(s_dev, dev(tok["x"], "bf16"), dev(tok["dt"]), dev(A),
                               dev(tok["B"], "bf16"), dev(tok["C"], "bf16"), dev(D))
    torch.cuda.synchronize()
    y_ref, s_ref = _oracle_steps(state, tok, A, D)
    assert rel(host(y), y_ref) <= TOL["bf16"]
    got, want = host(s_dev), oracle.round_bf16(s_ref)
    assert rel(got, s_ref) <= 4e-3
    # nearly every element is the correctly rounded fp64 state
    assert np.mean(got == want) >= 0.99


def test_multi_token_decode_with_dt_transform_and_gate():
    import state_space_model_chunked_gb300 as ssd
    b, T, H, P, N, G = 2, 20, 6, 64, 64, 3
    state = gen.decode_state(b, H, P, N, seed=13)
    A, D = gen.decode_params(H, seed=13)
    tok = _tokens(b, T, H, P, N, G, "bf16", 13)
    rng = np.random.default_rng(13)
    raw = rng.normal(-3.0, 1.5, size=tok["dt"].shape).astype(np.float32)
    tok["dt"] = raw
    bias = rng.normal(0.0, 0.5, size=(H,)).astype(np.float32)
    z = gen.bf16_round(rng.standard_normal((b, T, H, P)).astype(np.float32))[0]
    s_dev = dev(state)
    y = ssd.state_update_multi(s_dev, dev(tok["x"], "bf16"), dev(raw), dev(A),
                               dev(tok["B"], "bf16"), dev(tok["C"], "bf16"), dev(D),
                               dt_bias=dev(bias), dt_softplus=True, dt_limit=(1e-4, 0.5),
                               z=dev(z, "bf16"))
    torch.cuda.synchronize()
    kw = dict(bias=bias, softplus=True, lo=1e-4, hi=0.5)
    y_ref, s_ref = _oracle_steps(state, tok, A, D, dt_kw=kw, z=z)
    assert rel(host(y), y_ref) <= TOL["bf16"]
    assert rel(host(s_dev), s_ref) <= 1e-5


@pytest.mark.parametrize("scale", [1.0, 40.0, 300.0, -0.5])
def test_multi_token_decode_strong_decay_and_growth(scale):
    """Step sizes scaled so that a group of tokens decays by hundreds of
    e-folds (the scaled state is restored before it leaves fp32's range) or,
    with a negative scale, grows: the state and y still follow the chained
    steps."""
    import state_space_model_chunked_gb300 as ssd
    b, T, H, P, N, G = 2, 24, 4, 64, 128, 2
    state = gen.decode_state(b, H, P, N, seed=21)
    A, D = gen.decode_params(H, seed=21)
    tok = _tokens(b, T, H, P, N, G, "bf16", 21)
    tok["dt"] = (tok["dt"] * scale).astype(np.float32)
    s_dev = dev(state)
    y = ssd.state_update_multi(s_dev, dev(tok["x"], "bf16"), dev(tok["dt"]), dev(A),
                               dev(tok["B"], "bf16"), dev(tok["C"], "bf16"), dev(D))
    torch.cuda.synchronize()
    y_ref, s_ref = _oracle_steps(state, tok, A, D)
    assert rel(host(y), y_ref) <= TOL["bf16"]
    assert rel(host(s_dev), s_ref) <= 1e-5
