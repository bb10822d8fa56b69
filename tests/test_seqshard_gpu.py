"""One sequence split over GPUs by tokens, on one GPU: the range log-decay
and the state chain against fp64 numpy, and the whole decomposition -- each
range scanned from a zero state, the (log-decay, state) pairs chained, each
range scanned again from its entering state -- run through the library for
every range in turn (the ranks' all-gather becomes a Python list) and
compared with the fp64 oracle's scan of the unsplit sequence."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_chunked_gb300 import inputs as gen
from state_space_model_chunked_gb300.sharding import token_range
from tests.gpu_util import TOL, dev, host, rel

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("b,L,H", [(1, 1, 1), (2, 300, 5), (1, 65536, 80), (3, 1000, 40)])
@pytest.mark.parametrize("transform", [False, True])
def test_range_log_decay_matches_fp64_sum(b, L, H, transform):
    import state_space_model_chunked_gb300 as ssd
    inp = gen.scan_inputs(b, L, H, 8, 8, 1, "f32", seed=L + H)
    kw, d = {}, inp["dt"].astype(np.float64)
    if transform:
        rng = np.random.default_rng(L)
        raw = rng.normal(-3.0, 1.0, size=inp["dt"].shape).astype(np.float32)
        bias = rng.normal(0.0, 0.5, size=(H,)).astype(np.float32)
        inp["dt"] = raw
        kw = dict(dt_bias=dev(bias), dt_softplus=True, dt_limit=(1e-4, 0.2))
        d = oracle.dt_transform(raw, bias, True, 1e-4, 0.2)
    got = host(ssd.range_log_decay(dev(inp["dt"]), dev(inp["A"]), **kw))
    want = inp["A"].astype(np.float64)[None, :] * d.sum(axis=1)
    np.testing.assert_allclose(got, want, rtol=2e-6, atol=1e-6)


@pytest.mark.parametrize("R,with_init", [(1, False), (3, True), (8, True)])
def test_chain_states_matches_fp64_chain(R, with_init):
    import state_space_model_chunked_gb300 as ssd
    rng = np.random.default_rng(R)
    b, H, P, N = 2, 6, 16, 32
    contrib = rng.standard_normal((R, b, H, P, N)).astype(np.float32)
    decays = -rng.uniform(0.0, 5.0, size=(R, b, H)).astype(np.float32)
    init = rng.standard_normal((b, H, P, N)).astype(np.float32) if with_init else None
    got = host(ssd.chain_states(dev(contrib), dev(decays), dev(init)))
    h = np.zeros((b, H, P, N)) if init is None else init.astype(np.float64)
    for r in range(R):
        np.testing.assert_allclose(got[r], h, rtol=1e-5, atol=1e-5)
        h = np.exp(decays[r].astype(np.float64))[:, :, None, None] * h + contrib[r]


def _split_scan(inp, ranks, dtype, algo, heads=None):
    """The decomposition through the library, one range after another."""
    import state_space_model_chunked_gb300 as ssd
    L = inp["x"].shape[1]
    cuts = [token_range(L, ranks, r) for r in range(ranks)]
    A, D, init = dev(inp["A"]), dev(inp["D"]), dev(inp["init"])
    parts = [{k: dev(np.ascontiguousarray(inp[k][:, t0:t1]), dtype if k in ("x", "B", "C")
                     else "f32") for k in ("x", "dt", "B", "C")} for t0, t1 in cuts]
    contribs, decays = [], []
    for p in parts:
        _, f = ssd.scan_fwd(p["x"], p["dt"], A, p["B"], p["C"], D, 256, None, algo=algo)
        contribs.append(f)
        decays.append(ssd.range_log_decay(p["dt"], A))
    entering = ssd.chain_states(torch.stack(contribs), torch.stack(decays), init)
    ys, fin = [], None
    for r, p in enumerate(parts):
        y, fin = ssd.scan_fwd(p["x"], p["dt"], A, p["B"], p["C"], D, 256,
                              entering[r].contiguous(), algo=algo)
        ys.append(y)
    torch.cuda.synchronize()
    return host(torch.cat(ys, dim=1)), host(fin)


@pytest.mark.parametrize("b,L,H,G,ranks,algo,dtype", [
    (2, 5000, 8, 2, 3, 2, "bf16"),      # tensor-core path, ragged last range
    (1, 3000, 4, 1, 4, 2, "bf16"),
    (2, 700, 3, 1, 2, 1, "f32"),        # SIMT path
])
def test_token_split_matches_unsplit_oracle(b, L, H, G, ranks, algo, dtype):
    inp = gen.scan_inputs(b, L, H, 64, 128, G, dtype, seed=L + ranks, random_init=True)
    y, f = _split_scan(inp, ranks, dtype, algo)
    yr, fr = oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["init"])
    assert rel(y, yr) <= TOL[dtype] and rel(f, fr) <= TOL[dtype], (rel(y, yr), rel(f, fr))


def test_long_layer_split_over_four_ranges():
    """The 2.7B-shaped 65536-token layer as four ranges of 16384 tokens; four
    whole heads are checked against the oracle's unsplit scan."""
    s = gen.SCAN_SHAPES["mamba2_2p7b_L65536"]
    inp = gen.scan_inputs(s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups, "bf16",
                          seed=5, random_init=True)
    y, f = _split_scan(inp, 4, "bf16", 0)
    heads = [0, 17, 42, 79]
    yr, fr = oracle.scan_seq(inp["x"][:, :, heads], inp["dt"][:, :, heads], inp["A"][heads],
                             inp["B"], inp["C"], inp["D"][heads], inp["init"][:, heads])
    assert rel(y[:, :, heads], yr) <= TOL["bf16"]
    assert rel(f[:, heads], fr) <= TOL["bf16"]
