"""GPU parity of the chunked SSD scan (ssd_scan_fwd) against the fp64 oracle,
through the C ABI: every kernel path, the workloads' shapes, ragged and
degenerate edges."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_chunked_gb300 import inputs as gen
from tests.gpu_util import TOL, dev, host, rel, scan_on_gpu, scan_oracle

pytestmark = pytest.mark.gpu

AUTO, SIMT, TC = 0, 1, 2


def _check(inp, dtype, chunk, algo, tol=None):
    y, f = scan_on_gpu(inp, dtype, chunk, algo)
    yr, fr = scan_oracle(inp)
    tol = TOL[dtype] if tol is None else tol
    ey, ef = rel(y, yr), rel(f, fr)
    assert ey <= tol and ef <= tol, (ey, ef)
    return ey, ef


def test_fp32_workload_L256_H4_P64_N64():
    s = gen.SCAN_SHAPES["ssd_fp32_L256_H4_P64_N64"]
    inp = gen.scan_inputs_for(s, seed=0)
    _check(inp, "f32", s.chunk, AUTO)


@pytest.mark.parametrize("b,L,H,P,N,G", [
    (1, 1, 1, 16, 16, 1),        # one token
    (2, 200, 3, 16, 16, 1),      # ragged last tile
    (1, 130, 6, 20, 32, 3),      # ragged state-row block, several groups
    (3, 64, 4, 64, 64, 2),
    (1, 257, 2, 64, 128, 1),
    (1, 96, 2, 8, 256, 1),       # widest supported state
])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_init", [False, True])
def test_simt_path_shapes(b, L, H, P, N, G, dtype, with_init):
    inp = gen.scan_inputs(b, L, H, P, N, G, dtype, seed=L + N + b, random_init=with_init)
    _check(inp, dtype, 64, SIMT)


def test_simt_without_skip_term():
    inp = gen.scan_inputs(2, 100, 4, 32, 64, 2, "f32", seed=8, with_D=False)
    _check(inp, "f32", 32, SIMT)


@pytest.mark.parametrize("name", ["mamba2_130m_L4096", "mamba2_370m_b8_L2048"])
def test_prefill_workloads_full(name):
    s = gen.SCAN_SHAPES[name]
    inp = gen.scan_inputs_for(s, seed=0)
    _check(inp, s.dtype, s.chunk, AUTO)


@pytest.mark.parametrize("chunk", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("algo", [TC, SIMT])
def test_every_chunk_value_matches_oracle(chunk, algo):
    """`chunk` is validated and does not size the kernels' tiles: every
    allowed value gives the oracle's result on both kernel paths."""
    inp = gen.scan_inputs(1, 512, 4, 64, 128, 1, "bf16", seed=12, random_init=True)
    _check(inp, "bf16", chunk, algo)


# ---------------------------------------------------------------- tensor-core path
@pytest.mark.parametrize("b,L,H,G,with_init", [
    (1, 128, 2, 1, False),        # one tile, one head pair
    (1, 200, 2, 1, True),         # ragged last tile
    (1, 1, 2, 1, True),           # one token
    (2, 384, 4, 2, True),         # two groups, head pairs inside each
    (1, 256, 3, 1, False),        # odd heads per group: one head per CTA
    (1, 1000, 6, 3, True),        # odd heads per group, ragged, several groups
    (3, 640, 8, 1, True),         # batch > 1
])
def test_tc_path_matches_oracle(b, L, H, G, with_init):
    inp = gen.scan_inputs(b, L, H, 64, 128, G, "bf16", seed=L + H + b, random_init=with_init)
    _check(inp, "bf16", 128, TC)


def test_tc_path_many_segments():
    """A long sequence split across many CTAs: segment contributions, their
    chaining into entering states, and the scan from them."""
    inp = gen.scan_inputs(1, 8192, 2, 64, 128, 1, "bf16", seed=99, random_init=True)
    _check(inp, "bf16", 256, TC)


@pytest.mark.parametrize("b,H,G", [(4, 8, 2), (2, 16, 1)])
def test_tc_path_many_segments_four_heads_per_group(b, H, G):
    """Groups of four or more heads with enough segments (64 here) that the
    segment contributions are computed four heads per CTA over one shared B
    tile."""
    inp = gen.scan_inputs(b, 8192, H, 64, 128, G, "bf16", seed=41 + G, random_init=True)
    _check(inp, "bf16", 256, TC)


def test_tc_path_48_heads_two_groups_32k_tokens():
    """48 heads in two groups over 32768 tokens: 19 segments of 14 tiles, four
    heads per segment-kernel CTA, head pairs in the scan kernel.  The oracle
    checks six whole heads across both groups."""
    inp = gen.scan_inputs(1, 32768, 48, 64, 128, 2, "bf16", seed=77, random_init=True)
    y, f = scan_on_gpu(inp, "bf16", 256, TC)
    heads = [0, 5, 23, 24, 30, 47]
    g = [h // 24 for h in heads]
    yr, fr = oracle.scan_seq(inp["x"][:, :, heads], inp["dt"][:, :, heads], inp["A"][heads],
                             inp["B"][:, :, g], inp["C"][:, :, g], inp["D"][heads],
                             inp["init"][:, heads])
    assert rel(y[:, :, heads], yr) <= 1e-2
    assert rel(f[:, heads], fr) <= 1e-2


@pytest.mark.parametrize("scale", [20.0, 200.0])
def test_tc_path_strong_decay(scale):
    """Step sizes up to 2 (or 20) with |A| up to 16: the decay across one
    32-token block reaches hundreds of e-folds, beyond the factored mask's
    range, so diagonal blocks take the one-exponential-per-element form and
    long stretches of the state underflow to zero."""
    inp = gen.scan_inputs(2, 700, 4, 64, 128, 2, "bf16", seed=23, random_init=True)
    inp["dt"] = (inp["dt"] * scale).astype(np.float32)
    _check(inp, "bf16", 256, TC)


@pytest.mark.parametrize("algo", [TC, AUTO, SIMT])
def test_zero_and_negative_step_sizes(algo):
    """A fifth of the step sizes exactly 0 (that token neither decays the
    state nor adds to it) and a tenth small and negative (growth): every path,
    the default one included, follows the recurrence for any sign of dt."""
    inp = gen.scan_inputs(1, 700, 4, 64, 128, 2, "bf16", seed=31, random_init=True)
    dt = inp["dt"].astype(np.float64)
    m = np.random.default_rng(3).random(dt.shape)
    dt[m < 0.2] = 0.0
    dt[(m >= 0.2) & (m < 0.3)] *= -0.5
    inp["dt"] = dt.astype(np.float32)
    assert (inp["dt"] == 0).any() and (inp["dt"] < 0).any()
    _check(inp, "bf16", 256, algo)


def test_tc_path_without_skip():
    inp = gen.scan_inputs(1, 512, 4, 64, 128, 1, "bf16", seed=7, with_D=False)
    _check(inp, "bf16", 256, TC)


def test_tc_matches_simt():
    inp = gen.scan_inputs(2, 777, 4, 64, 128, 1, "bf16", seed=17, random_init=True)
    y1, f1 = scan_on_gpu(inp, "bf16", 256, TC)
    y2, f2 = scan_on_gpu(inp, "bf16", 256, SIMT)
    assert rel(y1, y2) <= 1e-2 and rel(f1, f2) <= 1e-2


def test_tc_reports_no_device_error():
    import state_space_model_chunked_gb300 as ssd
    inp = gen.scan_inputs(1, 300, 2, 64, 128, 1, "bf16", seed=3)
    scan_on_gpu(inp, "bf16", 64, TC)
    ssd.last_device_error()   # raises on a timed-out wait or misaligned carve-out


def test_long_context_2p7b_sampled_heads():
    """The 2.7B-shaped long-context layer (L=65536, 80 heads) at full size in
    the launch the benchmark times; the oracle checks four whole heads (every
    head is an independent recurrence)."""
    s = gen.SCAN_SHAPES["mamba2_2p7b_L65536"]
    inp = gen.scan_inputs_for(s, seed=0)
    y, f = scan_on_gpu(inp, "bf16", s.chunk, AUTO)
    heads = [0, 17, 42, 79]
    sub = {k: (v[:, :, heads] if k in ("x", "dt") else v) for k, v in inp.items()}
    sub["A"] = inp["A"][heads]
    sub["D"] = inp["D"][heads]
    yr, fr = oracle.scan_seq(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], sub["D"], None)
    assert rel(y[:, :, heads], yr) <= 1e-2
    assert rel(f[:, heads], fr) <= 1e-2


def test_profile_events_hook_eager_and_in_graph():
    """The profiling hook times the y-writing kernel both in eager launches and
    inside a captured CUDA graph, without changing the result."""
    import state_space_model_chunked_gb300 as ssd
    inp = gen.scan_inputs(1, 2048, 4, 64, 128, 1, "bf16", seed=5, random_init=True)
    x, Bm, Cm = dev(inp["x"], "bf16"), dev(inp["B"], "bf16"), dev(inp["C"], "bf16")
    dt, A, D, init = dev(inp["dt"]), dev(inp["A"]), dev(inp["D"]), dev(inp["init"])
    ws = torch.empty(max(ssd.scan_workspace_bytes(1, 2048, 4, 64, 128, 1, 256), 1),
                     dtype=torch.uint8, device=x.device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e1.record()
    torch.cuda.synchronize()
    ssd.scan_profile_events(e0, e1)
    y_eager, f_eager = ssd.scan_fwd(x, dt, A, Bm, Cm, D, 256, init, workspace=ws)
    ssd.scan_profile_events(None, None)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0
    y = torch.empty_like(x)
    f = torch.empty_like(f_eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ssd.scan_profile_events(e0, e1)
        ssd.scan_fwd(x, dt, A, Bm, Cm, D, 256, init, y=y, final_state=f, workspace=ws)
        ssd.scan_profile_events(None, None)
    g.replay()
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0
    assert torch.equal(y, y_eager) and torch.equal(f, f_eager)


def test_host_pipeline_matches_device_calls():
    """Host-buffer calls through HostScanPipeline (copies of consecutive calls
    overlapped, staging slots reused) give exactly the results of the same
    scans run on device tensors."""
    import state_space_model_chunked_gb300 as ssd
    pipe = ssd.HostScanPipeline(depth=2)
    cases, outs = [], []
    for i in range(5):
        inp = gen.scan_inputs(1, 1024, 4, 64, 128, 1, "bf16", seed=300 + i, random_init=True)
        host = {k: (torch.from_numpy(v).to(torch.bfloat16) if k in ("x", "B", "C")
                    else torch.from_numpy(v)).pin_memory() for k, v in inp.items()}
        out = (torch.empty(host["x"].shape, dtype=torch.bfloat16, pin_memory=True),
               torch.empty(host["init"].shape, dtype=torch.float32, pin_memory=True))
        pipe.submit(host["x"], host["dt"], host["A"], host["B"], host["C"], host["D"], 256,
                    host["init"], out=out)
        cases.append(host)
        outs.append(out)
    pipe.synchronize()
    for host, (yh, fh) in zip(cases, outs):
        d = {k: v.cuda() for k, v in host.items()}
        y, f = ssd.scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 256, d["init"])
        torch.cuda.synchronize()
        assert torch.equal(yh, y.cpu()) and torch.equal(fh, f.cpu())


# --------------------------------------------------------- dt transform fused
def _raw_dt_case(b, L, H, G, dtype, seed):
    """Inputs whose dt is a raw projection output (about N(-3, 1)), a per-head
    bias, and the fp64 step the transform makes of them."""
    inp = gen.scan_inputs(b, L, H, 64, 128, G, dtype, seed=seed, random_init=True)
    rng = np.random.default_rng(seed)
    inp["dt"] = rng.normal(-3.0, 1.0, size=inp["dt"].shape).astype(np.float32)
    bias = rng.uniform(-1.0, 1.0, size=(H,)).astype(np.float32)
    return inp, bias


@pytest.mark.parametrize("algo,dtype", [(TC, "bf16"), (SIMT, "f32"), (SIMT, "bf16")])
@pytest.mark.parametrize("limit", [None, (1e-3, 0.08)])
def test_scan_dt_softplus_bias_clamp(algo, dtype, limit):
    """dt <- clamp(softplus(dt_raw + bias), lo, hi) computed inside the kernels
    matches the oracle run on the fp64 transform of the same raw values."""
    inp, bias = _raw_dt_case(2, 700, 4, 2, dtype, seed=61)
    kw = dict(dt_bias=bias, dt_softplus=True, dt_limit=limit)
    y, f = scan_on_gpu(inp, dtype, 256, algo, **kw)
    lo, hi = limit if limit else (-np.inf, np.inf)
    ref = dict(inp, dt=oracle.dt_transform(inp["dt"], bias, True, lo, hi))
    yr, fr = scan_oracle(ref)
    tol = TOL[dtype]
    assert rel(y, yr) <= tol and rel(f, fr) <= tol, (rel(y, yr), rel(f, fr))


def test_scan_dt_transform_rejects_inverted_limits():
    import state_space_model_chunked_gb300 as ssd
    inp, bias = _raw_dt_case(1, 128, 2, 1, "bf16", seed=62)
    with pytest.raises(ssd.SsdError) as e:
        scan_on_gpu(inp, "bf16", 128, AUTO, dt_softplus=True, dt_limit=(1.0, 0.5))
    assert e.value.code == 1



# ---------------------------------------------------------------- packed sequences
def _varlen_on_gpu(inp, dtype, algo, chunk=256, **dt_kw):
    import state_space_model_chunked_gb300 as ssd
    if dt_kw.get("dt_bias") is not None:
        dt_kw = dict(dt_kw, dt_bias=dev(dt_kw["dt_bias"]))
    y, f = ssd.scan_fwd_varlen(dev(inp["x"], dtype), dev(inp["dt"]), dev(inp["A"]),
                               dev(inp["B"], dtype), dev(inp["C"], dtype), inp["cu"],
                               dev(inp["D"]), chunk, dev(inp["init"]), algo=algo, **dt_kw)
    torch.cuda.synchronize()
    return host(y), host(f)


def _check_varlen(inp, dtype, algo, dt=None, **dt_kw):
    """Whole-output and per-sequence relative L2 against the oracle (so the
    error of a short sequence is not hidden by the long ones)."""
    y, f = _varlen_on_gpu(inp, dtype, algo, **dt_kw)
    d = inp["dt"] if dt is None else dt
    yr, fr = oracle.scan_varlen(inp["x"], d, inp["A"], inp["B"], inp["C"], inp["cu"],
                                inp["D"], inp["init"])
    tol = TOL[dtype]
    assert rel(y, yr) <= tol and rel(f, fr) <= tol, (rel(y, yr), rel(f, fr))
    cu = inp["cu"]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if a < b:
            assert rel(y[a:b], yr[a:b]) <= tol, (s, rel(y[a:b], yr[a:b]))
        assert rel(f[s], fr[s]) <= tol, (s, rel(f[s], fr[s]))


@pytest.mark.parametrize("lengths,H,G,with_init", [
    ([1, 127, 128, 129, 1000, 5000], 4, 1, True),    # ragged tails; long one split
    ([300, 0, 2], 2, 1, True),                        # empty sequence in the middle
    ([128] * 8, 4, 2, False),                         # tile-aligned boundaries
    ([5000, 3], 3, 1, True),                          # odd heads per group
    ([700, 64, 1, 2000, 333], 8, 1, False),           # four heads per group
])
@pytest.mark.parametrize("algo", [TC, SIMT])
def test_varlen_matches_oracle(lengths, H, G, with_init, algo):
    inp = gen.varlen_inputs(lengths, H, 64, 128, G, "bf16", seed=sum(lengths) + H,
                            random_init=with_init)
    _check_varlen(inp, "bf16", algo)


def test_varlen_many_short_sequences():
    """More sequences than the offset-table kernel's block (1024) walks at
    once; lengths 1..40 tokens."""
    lengths = gen.packed_lengths(2500, 1, 40, seed=3)
    inp = gen.varlen_inputs(lengths, 2, 64, 128, 1, "bf16", seed=4, random_init=True)
    _check_varlen(inp, "bf16", TC)


def test_varlen_2p7b_heads_mixed_lengths():
    """The 80-head model's shape on a packed batch of 16 log-uniform lengths
    in [64, 8192] tokens."""
    lengths = gen.packed_lengths(16, 64, 8192, seed=11)
    inp = gen.varlen_inputs(lengths, 80, 64, 128, 1, "bf16", seed=12, random_init=True)
    _check_varlen(inp, "bf16", AUTO)


def test_varlen_dt_transform():
    inp = gen.varlen_inputs([900, 17, 2100], 4, 64, 128, 1, "bf16", seed=21, random_init=True)
    rng = np.random.default_rng(22)
    inp["dt"] = rng.normal(-3.0, 1.0, size=inp["dt"].shape).astype(np.float32)
    bias = rng.normal(0.0, 0.5, size=(4,)).astype(np.float32)
    d = oracle.dt_transform(inp["dt"], bias, True, 1e-3, 0.2)
    _check_varlen(inp, "bf16", TC, dt=d, dt_bias=bias, dt_softplus=True, dt_limit=(1e-3, 0.2))


def test_varlen_without_tokens_returns_initial_states():
    import state_space_model_chunked_gb300 as ssd
    inp = gen.varlen_inputs([0, 0, 0], 2, 64, 128, 1, "bf16", seed=1, random_init=True)
    y, f = _varlen_on_gpu(inp, "bf16", AUTO)
    assert y.shape == (0, 2, 64)
    np.testing.assert_array_equal(f, inp["init"])
    with pytest.raises(ssd.SsdError):
        _varlen_on_gpu(inp, "bf16", TC)


def test_varlen_one_sequence_matches_batched_call():
    inp = gen.scan_inputs(1, 3000, 4, 64, 128, 1, "bf16", seed=9, random_init=True)
    yb, fb = scan_on_gpu(inp, "bf16", 256, TC)
    packed = {k: (v[0] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    packed["cu"] = np.array([0, 3000], np.int32)
    yv, fv = _varlen_on_gpu(packed, "bf16", TC)
    assert rel(yv, yb[0]) <= 1e-3 and rel(fv, fb) <= 1e-3


# ---------------------------------------------------------------- output gate
@pytest.mark.parametrize("b,L,H,G,algo,dtype", [
    (1, 1000, 4, 1, TC, "bf16"),        # ragged last tile
    (2, 640, 6, 3, TC, "bf16"),         # one head per CTA, batch 2
    (1, 4096, 24, 1, AUTO, "bf16"),     # the 130M layer
    (2, 300, 4, 2, SIMT, "f32"),
    (1, 200, 3, 1, SIMT, "bf16"),
])
def test_output_gate_matches_oracle(b, L, H, G, algo, dtype):
    inp = gen.scan_inputs(b, L, H, 64, 128, G, dtype, seed=L + H, random_init=True)
    z = gen.gate_input((b, L, H, 64), dtype, seed=L)
    y, f = scan_on_gpu(inp, dtype, 256, algo, z=dev(z, dtype))
    yr, fr = scan_oracle(inp)
    assert rel(y, oracle.gate(yr, z)) <= TOL[dtype], rel(y, oracle.gate(yr, z))
    assert rel(f, fr) <= TOL[dtype]


def test_output_gate_with_dt_transform_long():
    """Gate and dt transform together on a sequence long enough to be split
    into segments (chained states), 8 heads."""
    inp = gen.scan_inputs(1, 20000, 8, 64, 128, 1, "bf16", seed=31, random_init=True)
    rng = np.random.default_rng(31)
    raw = rng.normal(-4.0, 1.0, size=inp["dt"].shape).astype(np.float32)
    bias = rng.normal(0.0, 0.5, size=(8,)).astype(np.float32)
    z = gen.gate_input(inp["x"].shape, "bf16", seed=31)
    d = oracle.dt_transform(raw, bias, True, 1e-4, 0.1)
    inp_raw = dict(inp, dt=raw)
    y, f = scan_on_gpu(inp_raw, "bf16", 256, TC, dt_bias=bias, dt_softplus=True,
                       dt_limit=(1e-4, 0.1), z=dev(z, "bf16"))
    yr, fr = oracle.scan_seq(inp["x"], d, inp["A"], inp["B"], inp["C"], inp["D"], inp["init"])
    assert rel(y, oracle.gate(yr, z)) <= 1e-2 and rel(f, fr) <= 1e-2


@pytest.mark.parametrize("algo", [TC, SIMT])
def test_varlen_output_gate(algo):
    inp = gen.varlen_inputs([1, 300, 129, 2000], 4, 64, 128, 1, "bf16", seed=41,
                            random_init=True)
    z = gen.gate_input(inp["x"].shape, "bf16", seed=41)
    y, f = _varlen_on_gpu(inp, "bf16", algo, z=dev(z, "bf16"))
    yr, fr = oracle.scan_varlen(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["cu"],
                                inp["D"], inp["init"])
    assert rel(y, oracle.gate(yr, z)) <= 1e-2 and rel(f, fr) <= 1e-2
    cu = inp["cu"]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        assert rel(y[a:b], oracle.gate(yr[a:b], z[a:b])) <= 1e-2


def test_varlen_long_sequence_four_head_segments():
    """A packed batch whose long sequence is split into segments at 80 heads:
    the segment-contribution kernel then takes four heads per CTA (the packed
    form of the long-context plan), next to short unsplit sequences."""
    inp = gen.varlen_inputs([20000, 300, 5], 80, 64, 128, 1, "bf16", seed=51, random_init=True)
    _check_varlen(inp, "bf16", TC)


def test_headline_workload_in_cuda_graph_sampled_heads():
    """The 2.7B-shaped 65536-token layer (80 heads, one group) exactly as the
    benchmark times it: inputs drawn on the device by the benchmark's own
    generator, the calls captured in a CUDA graph and replayed.  Three whole
    heads (first, middle, last; each an independent recurrence) are checked
    against the oracle, y and final state."""
    import sys
    import os
    import state_space_model_chunked_gb300 as ssd
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    shape = gen.SCAN_SHAPES["mamba2_2p7b_L65536"]
    device = torch.device("cuda")
    s = bench.make_scan_set(shape, 1234, device)
    ws = torch.empty(max(ssd.scan_workspace_bytes(shape.batch, shape.seqlen, shape.nheads,
                                                  shape.headdim, shape.dstate, shape.ngroups,
                                                  shape.chunk), 1),
                     dtype=torch.uint8, device=device)

    def call():
        ssd.scan_fwd(s["x"], s["dt"], s["A"], s["B"], s["C"], s["D"], shape.chunk, s["init"],
                     y=s["y"], final_state=s["final"], workspace=ws)

    call()                                    # outside capture (sets function attributes)
    torch.cuda.synchronize()
    s["y"].zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    g.replay()
    torch.cuda.synchronize()
    heads = [0, 41, 79]
    hx = host(s["x"][:, :, heads])
    yo, fo = oracle.scan_seq(hx, host(s["dt"][:, :, heads]), host(s["A"][heads]), host(s["B"]),
                             host(s["C"]), host(s["D"][heads]), None)
    assert rel(host(s["y"][:, :, heads]), yo) <= TOL["bf16"]
    assert rel(host(s["final"][:, heads]), fo) <= TOL["bf16"]
    ssd.last_device_error()
