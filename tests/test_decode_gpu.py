"""GPU parity of the decode state update (ssd_state_update) against the fp64
oracle's decode step, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_chunked_gb300 import inputs as gen
from tests.gpu_util import TOL, dev, host, rel

pytestmark = pytest.mark.gpu


def _one_step(b, H, P, N, G, dtype, seed=0, with_D=True):
    import state_space_model_chunked_gb300 as ssd
    state = gen.decode_state(b, H, P, N, seed=seed)
    A, D = gen.decode_params(H, seed=seed)
    if not with_D:
        D = None
    tok = gen.decode_token_inputs(b, H, P, N, G, dtype, seed=seed, step=0)
    s_dev = dev(state)
    y = ssd.state_update(s_dev, dev(tok["x"], dtype), dev(tok["dt"]), dev(A),
                         dev(tok["B"], dtype), dev(tok["C"], dtype), dev(D))
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.step(state, tok["x"], tok["dt"], A, tok["B"], tok["C"], D)
    return host(y), host(s_dev), y_ref, s_ref


@pytest.mark.parametrize("b,H,P,N,G", [
    (3, 4, 16, 16, 2), (2, 80, 64, 128, 1), (1, 3, 1, 4, 1), (2, 6, 7, 8, 3),
    (2, 4, 64, 256, 1), (5, 2, 33, 64, 2), (1, 1, 64, 32, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_matches_oracle(b, H, P, N, G, dtype):
    y, s, y_ref, s_ref = _one_step(b, H, P, N, G, dtype, seed=b * 100 + N)
    assert rel(y, y_ref) <= TOL[dtype], rel(y, y_ref)
    assert rel(s, s_ref) <= TOL[dtype], rel(s, s_ref)
    # the state update itself is fp32 FMA on exact inputs in both dtypes
    assert rel(s, s_ref) <= 1e-6


def test_decode_without_skip():
    y, s, y_ref, s_ref = _one_step(2, 8, 64, 128, 2, "bf16", seed=5, with_D=False)
    assert rel(y, y_ref) <= 1e-2 and rel(s, s_ref) <= 1e-6


def test_decode_many_steps_2p7b_layer():
    """128 consecutive tokens of one Mamba-2-2.7B-shaped layer (H80 P64 N128),
    batch 2: y at every step and the final state track the oracle."""
    import state_space_model_chunked_gb300 as ssd
    b, H, P, N, G = 2, 80, 64, 128, 1
    state = gen.decode_state(b, H, P, N, seed=3)
    A, D = gen.decode_params(H, seed=3)
    s_dev = dev(state)
    s_ref = state.astype(np.float64)
    worst = 0.0
    for t in range(128):
        tok = gen.decode_token_inputs(b, H, P, N, G, "bf16", seed=3, step=t)
        y = ssd.state_update(s_dev, dev(tok["x"], "bf16"), dev(tok["dt"]), dev(A),
                             dev(tok["B"], "bf16"), dev(tok["C"], "bf16"), dev(D))
        y_ref, s_ref = oracle.step(s_ref, tok["x"], tok["dt"], A, tok["B"], tok["C"], D)
        worst = max(worst, rel(host(y), y_ref))
    assert worst <= 1e-2
    assert rel(host(s_dev), s_ref) <= 1e-4


def test_decode_full_stack_sampled():
    """The 64-layer stack at batch 16, flattened as (layer, head) heads with
    one group per layer -- the launch the benchmark times.  The oracle checks
    a sample of (batch, layer) slices, each an independent recurrence."""
    import state_space_model_chunked_gb300 as ssd
    layers, H, P, N = 64, 80, 64, 128
    b = 16
    Hf, G = layers * H, layers
    state = gen.device_decode_state(b, Hf, P, N, seed=1)
    A, D = gen.decode_params(Hf, seed=1)
    tok = gen.device_decode_token_inputs(b, Hf, P, N, G, seed=1, step=0)
    before = {}
    samples = [(0, 0), (3, 17), (15, 63), (9, 40)]
    for (bi, li) in samples:
        before[(bi, li)] = state[bi, li * H:(li + 1) * H].double().cpu().numpy()
    y = ssd.state_update(state, tok["x"], tok["dt"], dev(A), tok["B"], tok["C"], dev(D))
    torch.cuda.synchronize()
    for (bi, li) in samples:
        hs = slice(li * H, (li + 1) * H)
        x = tok["x"][bi:bi + 1, hs].float().cpu().numpy()
        dt = tok["dt"][bi:bi + 1, hs].cpu().numpy()
        Bg = tok["B"][bi:bi + 1, li:li + 1].float().cpu().numpy()
        Cg = tok["C"][bi:bi + 1, li:li + 1].float().cpu().numpy()
        y_ref, s_ref = oracle.step(before[(bi, li)][None], x, dt, A[hs], Bg, Cg, D[hs])
        assert rel(host(y[bi:bi + 1, hs]), y_ref) <= 1e-2
        assert rel(host(state[bi:bi + 1, hs]), s_ref) <= 1e-6


@pytest.mark.parametrize("N,dtype", [(128, "bf16"), (256, "bf16"), (64, "f32"), (16, "bf16")])
def test_decode_streaming_path_multi_step(N, dtype):
    """Enough (batch, head) states that every SM walks several of them through
    the shared-memory ring (the launch used for large decode stacks)."""
    import state_space_model_chunked_gb300 as ssd
    b, H, P, G = 8, 160, 64, 4
    state = gen.decode_state(b, H, P, N, seed=N)
    A, D = gen.decode_params(H, seed=N)
    s_dev = dev(state)
    s_ref = state.astype(np.float64)
    for t in range(3):
        tok = gen.decode_token_inputs(b, H, P, N, G, dtype, seed=N, step=t)
        y = ssd.state_update(s_dev, dev(tok["x"], dtype), dev(tok["dt"]), dev(A),
                             dev(tok["B"], dtype), dev(tok["C"], dtype), dev(D))
        y_ref, s_ref = oracle.step(s_ref, tok["x"], tok["dt"], A, tok["B"], tok["C"], D)
        assert rel(host(y), y_ref) <= TOL[dtype]
    assert rel(host(s_dev), s_ref) <= 1e-6
    ssd.last_device_error()


@pytest.mark.parametrize("units", [(3, 10), (8, 160)])     # classic and streaming launch
def test_decode_dt_softplus_bias(units):
    """The decode update with dt <- clamp(softplus(dt_raw + bias), lo, hi)
    computed in the kernel, against the oracle step on the fp64 transform."""
    import state_space_model_chunked_gb300 as ssd
    b, H = units
    P, N, G = 64, 128, 2
    state = gen.decode_state(b, H, P, N, seed=9)
    A, D = gen.decode_params(H, seed=9)
    tok = gen.decode_token_inputs(b, H, P, N, G, "bf16", seed=9, step=0)
    rng = np.random.default_rng(9)
    raw = rng.normal(-3.0, 1.0, size=(b, H)).astype(np.float32)
    bias = rng.uniform(-1.0, 1.0, size=(H,)).astype(np.float32)
    s_dev = dev(state)
    y = ssd.state_update(s_dev, dev(tok["x"], "bf16"), dev(raw), dev(A), dev(tok["B"], "bf16"),
                         dev(tok["C"], "bf16"), dev(D), dt_bias=dev(bias), dt_softplus=True,
                         dt_limit=(1e-3, 0.08))
    torch.cuda.synchronize()
    dt_eff = oracle.dt_transform(raw, bias, True, 1e-3, 0.08)
    y_ref, s_ref = oracle.step(state, tok["x"], dt_eff, A, tok["B"], tok["C"], D)
    assert rel(host(y), y_ref) <= 1e-2
    assert rel(host(s_dev), s_ref) <= 1e-6



@pytest.mark.parametrize("units,dtype", [((3, 10), "bf16"), ((8, 160), "bf16"),
                                         ((4, 6), "f32"), ((8, 160), "f32")])
def test_decode_output_gate(units, dtype):
    """y <- y * silu(z) in the kernel (classic and streaming launches), with
    and without the dt transform, against the oracle step and gate; the state
    is not touched by the gate."""
    import state_space_model_chunked_gb300 as ssd
    b, H = units
    P, N, G = 64, 128, 2
    state = gen.decode_state(b, H, P, N, seed=13)
    A, D = gen.decode_params(H, seed=13)
    tok = gen.decode_token_inputs(b, H, P, N, G, dtype, seed=13, step=0)
    z = gen.gate_input((b, H, P), dtype, seed=13)
    y_ref, s_ref = oracle.step(state, tok["x"], tok["dt"], A, tok["B"], tok["C"], D)
    s_dev = dev(state)
    y = ssd.state_update(s_dev, dev(tok["x"], dtype), dev(tok["dt"]), dev(A),
                         dev(tok["B"], dtype), dev(tok["C"], dtype), dev(D), z=dev(z, dtype))
    torch.cuda.synchronize()
    assert rel(host(y), oracle.gate(y_ref, z)) <= TOL[dtype]
    assert rel(host(s_dev), s_ref) <= 1e-6
    # with the dt transform as well
    raw = np.log(np.expm1(tok["dt"].astype(np.float64))).astype(np.float32)  # softplus^-1
    s_dev = dev(state)
    y = ssd.state_update(s_dev, dev(tok["x"], dtype), dev(raw), dev(A), dev(tok["B"], dtype),
                         dev(tok["C"], dtype), dev(D), dt_softplus=True, z=dev(z, dtype))
    torch.cuda.synchronize()
    d = oracle.dt_transform(raw, None, True)
    y_ref2, s_ref2 = oracle.step(state, tok["x"], d, A, tok["B"], tok["C"], D)
    assert rel(host(y), oracle.gate(y_ref2, z)) <= TOL[dtype]
    assert rel(host(s_dev), s_ref2) <= 1e-6


@pytest.mark.parametrize("units,steps", [((3, 10), 1), ((8, 160), 1), ((2, 12), 16),
                                         ((8, 160), 8)])
def test_decode_bf16_state(units, steps):
    """State stored as bfloat16 (classic and streaming launches): fp32 update,
    y from it, the state rounded to nearest even; against the oracle's
    bf16-state step chained over `steps` tokens.  One step must reproduce the
    oracle's rounded state exactly except for rare last-bit ties decided from
    fp32 instead of fp64 values."""
    import state_space_model_chunked_gb300 as ssd
    b, H = units
    P, N, G = 64, 128, 2
    st0 = gen.bf16_round(gen.decode_state(b, H, P, N, seed=17))[0]
    A, D = gen.decode_params(H, seed=17)
    s_dev = dev(st0, "bf16")
    s_ref = st0.astype(np.float64)
    for k in range(steps):
        tok = gen.decode_token_inputs(b, H, P, N, G, "bf16", seed=17, step=k)
        y = ssd.state_update(s_dev, dev(tok["x"], "bf16"), dev(tok["dt"]), dev(A),
                             dev(tok["B"], "bf16"), dev(tok["C"], "bf16"), dev(D))
        torch.cuda.synchronize()
        y_ref, s_ref = oracle.step_bf16_state(s_ref, tok["x"], tok["dt"], A, tok["B"], tok["C"],
                                              D)
        assert rel(host(y), y_ref) <= 1e-2, (k, rel(host(y), y_ref))
    s = host(s_dev)
    assert s_dev.dtype == torch.bfloat16
    assert rel(s, s_ref) <= 1e-2, rel(s, s_ref)
    if steps == 1:
        assert np.mean(s == s_ref) >= 0.99


def test_decode_bf16_state_needs_bf16_inputs():
    import state_space_model_chunked_gb300 as ssd
    b, H, P, N, G = 1, 2, 16, 16, 1
    s_dev = torch.zeros((b, H, P, N), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((b, H, P), device="cuda")
    with pytest.raises(ssd.SsdError):
        ssd.state_update(s_dev, x, torch.ones((b, H), device="cuda"),
                         torch.zeros(H, device="cuda"), torch.zeros((b, G, N), device="cuda"),
                         torch.zeros((b, G, N), device="cuda"))


@pytest.mark.parametrize("b,H,G", [(7, 91, 1), (5, 123, 3)])
def test_decode_bf16_state_streaming_odd_state_count(b, H, G):
    """bf16 states through the streaming kernel with an odd number of (batch,
    head) states (the ring's last stage holds a single state) and stages that
    cross batch rows and group boundaries."""
    import state_space_model_chunked_gb300 as ssd
    P, N = 64, 128
    st0 = gen.bf16_round(gen.decode_state(b, H, P, N, seed=29))[0]
    A, D = gen.decode_params(H, seed=29)
    s_dev = dev(st0, "bf16")
    tok = gen.decode_token_inputs(b, H, P, N, G, "bf16", seed=29, step=0)
    y = ssd.state_update(s_dev, dev(tok["x"], "bf16"), dev(tok["dt"]), dev(A),
                         dev(tok["B"], "bf16"), dev(tok["C"], "bf16"), dev(D))
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.step_bf16_state(st0, tok["x"], tok["dt"], A, tok["B"], tok["C"], D)
    assert rel(host(y), y_ref) <= 1e-2
    s = host(s_dev)
    assert rel(s, s_ref) <= 1e-2
    assert np.mean(s == s_ref) >= 0.99


@pytest.mark.parametrize("b,layers", [(1, 1), (1, 64), (16, 8)])
@pytest.mark.parametrize("in_graph", [False, True])
def test_chained_calls_see_the_previous_output(b, layers, in_graph):
    """Decode calls launched back to back, each reading the previous call's
    y as its x (x_{k+1} = y_k): the kernels may be scheduled while their
    predecessor runs, so each must wait for it before reading.  Eight calls,
    eagerly or captured in one CUDA graph, against the oracle stepping the same
    chain with the bf16 rounding of y between steps.  One layer of 80 heads at
    batch 1 takes the row-split single-state kernel; 64 layers at batch 1 the
    streaming kernel with programmatic launch, 8 layers at batch 16 (67 states
    per SM) the streaming kernel without it."""
    import state_space_model_chunked_gb300 as ssd
    H, P, N, G = 80 * layers, 64, 128, layers
    state = gen.decode_state(b, H, P, N, seed=7 + b)
    A, D = gen.decode_params(H, seed=7)
    toks = [gen.decode_token_inputs(b, H, P, N, G, "bf16", seed=7, step=k) for k in range(8)]
    s_dev = dev(state)
    ys = [torch.empty((b, H, P), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    x0 = dev(toks[0]["x"], "bf16")
    ins = [(dev(t["dt"]), dev(t["B"], "bf16"), dev(t["C"], "bf16")) for t in toks]
    A_d, D_d = dev(A), dev(D)

    def chain():
        x = x0
        for k in range(8):
            y = ys[k % 2]
            ssd.state_update(s_dev, x, ins[k][0], A_d, ins[k][1], ins[k][2], D_d, y=y)
            x = y

    if in_graph:
        s0 = s_dev.clone()
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            chain()                            # warm-up outside capture
            torch.cuda.synchronize()
            s_dev.copy_(s0)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                chain()
            torch.cuda.synchronize()
            s_dev.copy_(s0)
            torch.cuda.synchronize()
            g.replay()
        torch.cuda.synchronize()
    else:
        chain()
        torch.cuda.synchronize()
    s_ref, x = state.astype(np.float64), toks[0]["x"]
    for k in range(8):
        y_ref, s_ref = oracle.step(s_ref, x, toks[k]["dt"], A, toks[k]["B"], toks[k]["C"], D)
        x = oracle.round_bf16(y_ref)
    assert rel(host(s_dev), s_ref) <= TOL["bf16"], rel(host(s_dev), s_ref)
    assert rel(host(ys[1]), y_ref) <= TOL["bf16"], rel(host(ys[1]), y_ref)
