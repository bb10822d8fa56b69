"""GPU parity of fp8 (E4M3) prefill inputs against the fp64 oracle, through
the C ABI: the widening kernel bit for bit against the oracle's decode of
every code, and the scan on fp8 x/B/C -- tensor-core and SIMT paths, packed
sequences, the fused gate and dt transform, the 2.7B long-context layer --
against the oracle run on the decoded inputs.

The pages name reduced precision as future work ("Mamba-Family State-Space
Model Kernels on a Programmable CGLA", sections V.A and VI) and fix no
format or tolerance.  Every E4M3 value is a bfloat16 value, the library
widens exactly and then runs its bf16 path, so the bar is the bf16 path's
(relative L2 1e-2), and the result must equal the bf16 call on the widened
values bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_chunked_gb300 import inputs as gen
from tests.gpu_util import TOL, decoded, dev, host, rel, scan_on_gpu, scan_oracle

pytestmark = pytest.mark.gpu

AUTO, SIMT, TC = 0, 1, 2


def _check(inp, chunk, algo):
    y, f = scan_on_gpu(inp, "fp8", chunk, algo)
    yr, fr = scan_oracle(inp)
    ey, ef = rel(y, yr), rel(f, fr)
    assert ey <= TOL["fp8"] and ef <= TOL["fp8"], (ey, ef)
    return y, f


@pytest.mark.parametrize("n", [1, 7, 8, 15, 16, 256, 4096, 4096 + 13, 8 * 1024 + 3,
                               (1 << 20) + 7])
def test_widening_is_the_oracle_decode_bit_for_bit(n):
    """Every code (each of the 256 appears once before the random rest);
    lengths below, at and above one 8-value chunk and one CTA's 512 chunks,
    with and without a ragged tail: equal values, equal signs of zero, NaN at
    the NaN codes."""
    import state_space_model_chunked_gb300 as ssd
    rng = np.random.default_rng(n)
    codes = rng.integers(0, 256, size=n, dtype=np.uint8)
    codes[:min(n, 256)] = np.arange(min(n, 256), dtype=np.uint8)
    out = ssd.fp8_e4m3_to_bf16(torch.from_numpy(codes).cuda())
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref = oracle.decode_e4m3(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("b,L,H,G,with_init", [
    (1, 200, 2, 1, True),          # ragged last tile
    (2, 384, 4, 2, True),          # two groups
    (1, 1000, 6, 3, False),        # odd heads per group
    (1, 8192, 2, 1, True),         # many segments: contributions and chaining
    (2, 8192, 16, 1, True),        # four heads per segment-kernel CTA
])
def test_fp8_tc_path_matches_oracle(b, L, H, G, with_init):
    inp = gen.scan_inputs(b, L, H, 64, 128, G, "fp8", seed=L + H + 3, random_init=with_init)
    _check(inp, 256, TC)


@pytest.mark.parametrize("b,L,H,P,N,G", [
    (2, 200, 3, 16, 16, 1),
    (1, 130, 6, 20, 32, 3),        # headdim 20: rows not a multiple of 16 values
    (1, 77, 2, 8, 4, 1),           # every array shorter than a few vectors
])
def test_fp8_simt_path_matches_oracle(b, L, H, P, N, G):
    inp = gen.scan_inputs(b, L, H, P, N, G, "fp8", seed=L + P, random_init=True)
    _check(inp, 64, SIMT)


@pytest.mark.parametrize("algo", [TC, SIMT])
def test_fp8_equals_bf16_call_on_widened_values(algo):
    """The fp8 call is the bf16 call on the exactly widened inputs: y and the
    final state agree bit for bit."""
    inp = gen.scan_inputs(1, 3000, 4, 64, 128, 1, "fp8", seed=17, random_init=True)
    y8, f8 = scan_on_gpu(inp, "fp8", 256, algo)
    wide = decoded(inp)
    y16, f16 = scan_on_gpu(wide, "bf16", 256, algo)
    assert np.array_equal(y8, y16)
    assert np.array_equal(f8, f16)


@pytest.mark.parametrize("algo", [TC, SIMT])
def test_fp8_varlen_matches_oracle(algo):
    import state_space_model_chunked_gb300 as ssd
    inp = gen.varlen_inputs([1, 127, 129, 1000, 5000, 0, 3], 4, 64, 128, 1, "fp8", seed=29,
                            random_init=True)
    y, f = ssd.scan_fwd_varlen(dev(inp["x"], "fp8"), dev(inp["dt"]), dev(inp["A"]),
                               dev(inp["B"], "fp8"), dev(inp["C"], "fp8"), inp["cu"],
                               dev(inp["D"]), 256, dev(inp["init"]), algo=algo)
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16
    y, f = host(y), host(f)
    d = decoded(inp)
    yr, fr = oracle.scan_varlen(d["x"], d["dt"], d["A"], d["B"], d["C"], d["cu"], d["D"],
                                d["init"])
    assert rel(y, yr) <= TOL["fp8"] and rel(f, fr) <= TOL["fp8"], (rel(y, yr), rel(f, fr))
    cu = inp["cu"]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if a < b:
            assert rel(y[a:b], yr[a:b]) <= TOL["fp8"], s
        assert rel(f[s], fr[s]) <= TOL["fp8"], s


def test_fp8_with_gate_and_dt_transform():
    """fp8 x/B/C with the bf16 gate z and a softplus dt transform on a sequence
    split into segments."""
    inp = gen.scan_inputs(1, 9000, 8, 64, 128, 1, "fp8", seed=37, random_init=True)
    rng = np.random.default_rng(37)
    raw = rng.normal(-4.0, 1.0, size=inp["dt"].shape).astype(np.float32)
    bias = rng.normal(0.0, 0.5, size=(8,)).astype(np.float32)
    z = gen.gate_input(inp["x"].shape, "bf16", seed=37)
    y, f = scan_on_gpu(dict(inp, dt=raw), "fp8", 256, TC, dt_bias=bias, dt_softplus=True,
                       dt_limit=(1e-4, 0.1), z=dev(z, "bf16"))
    d = decoded(inp)
    yr, fr = oracle.scan_seq(d["x"], oracle.dt_transform(raw, bias, True, 1e-4, 0.1), d["A"],
                             d["B"], d["C"], d["D"], d["init"])
    assert rel(y, oracle.gate(yr, z)) <= TOL["fp8"] and rel(f, fr) <= TOL["fp8"]


def test_fp8_long_context_2p7b_sampled_heads():
    """The 2.7B-shaped long-context layer (L=65536, 80 heads) with fp8 inputs
    at full size, as the benchmark's fp8 line runs it; the oracle checks four
    whole heads on the decoded inputs."""
    s = gen.SCAN_SHAPES["mamba2_2p7b_L65536"]
    inp = gen.scan_inputs(s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups, "fp8",
                          seed=0)
    y, f = scan_on_gpu(inp, "fp8", s.chunk, AUTO)
    heads = [0, 17, 42, 79]
    d = decoded(dict(inp, x=inp["x"][:, :, heads]))
    yr, fr = oracle.scan_seq(d["x"], inp["dt"][:, :, heads], inp["A"][heads], d["B"], d["C"],
                             inp["D"][heads], None)
    assert rel(y[:, :, heads], yr) <= TOL["fp8"]
    assert rel(f[:, heads], fr) <= TOL["fp8"]


def test_fp8_decode_is_refused():
    import state_space_model_chunked_gb300 as ssd
    state = torch.zeros(1, 2, 16, 16, device="cuda")
    x = torch.zeros(1, 2, 16, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    B = torch.zeros(1, 1, 16, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    with pytest.raises(ssd.SsdError) as e:
        ssd.state_update(state, x, torch.zeros(1, 2, device="cuda"),
                         torch.zeros(2, device="cuda"), B, B)
    assert e.value.code == 2


def test_fp8_varlen_without_tokens_returns_initial_states():
    """A packed fp8 batch of empty sequences has no values to widen: the call
    gives each sequence its initial state, as for bf16."""
    import state_space_model_chunked_gb300 as ssd
    inp = gen.varlen_inputs([0, 0, 0], 2, 64, 128, 1, "fp8", seed=1, random_init=True)
    y, f = ssd.scan_fwd_varlen(dev(inp["x"], "fp8"), dev(inp["dt"]), dev(inp["A"]),
                               dev(inp["B"], "fp8"), dev(inp["C"], "fp8"), inp["cu"],
                               dev(inp["D"]), 256, dev(inp["init"]))
    torch.cuda.synchronize()
    assert y.shape == (0, 2, 64) and y.dtype == torch.bfloat16
    np.testing.assert_array_equal(host(f), inp["init"])
