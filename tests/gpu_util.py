"""Helpers shared by the GPU parity tests: move seeded numpy inputs to the
device in the dtype the workload names, and compare with the oracle."""
import numpy as np
import torch

import oracle

# relative L2 bars: fp32 / bf16-input / fp8-input workloads.  fp8 inputs are
# widened exactly to bfloat16 and take the bf16 path, so they share its bar.
TOL = {"f32": 1e-4, "bf16": 1e-2, "fp8": 1e-2}


def dev(a, dtype="f32"):
    """numpy float32 -> CUDA tensor; bf16 values are exactly representable so
    the conversion is exact.  dtype "fp8": `a` holds uint8 E4M3 codes, moved
    as a float8_e4m3fn tensor."""
    if a is None:
        return None
    if dtype == "fp8":
        codes = torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8))
        return codes.view(torch.float8_e4m3fn).cuda()
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.cuda()


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def scan_on_gpu(inp, dtype, chunk, algo=0, **dt_kw):
    import state_space_model_chunked_gb300 as ssd
    if dt_kw.get("dt_bias") is not None:
        dt_kw = dict(dt_kw, dt_bias=dev(dt_kw["dt_bias"]))
    y, fin = ssd.scan_fwd(dev(inp["x"], dtype), dev(inp["dt"]), dev(inp["A"]),
                          dev(inp["B"], dtype), dev(inp["C"], dtype), dev(inp["D"]),
                          chunk, dev(inp["init"]), algo=algo, **dt_kw)
    torch.cuda.synchronize()
    return host(y), host(fin)


def decoded(inp):
    """The inputs with fp8 x, B, C (uint8 E4M3 codes) replaced by the oracle's
    fp64 decode of them; other inputs unchanged."""
    out = dict(inp)
    for k in ("x", "B", "C"):
        if out.get(k) is not None and np.asarray(out[k]).dtype == np.uint8:
            out[k] = oracle.decode_e4m3(out[k])
    return out


def scan_oracle(inp):
    inp = decoded(inp)
    return oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                           inp["D"], inp["init"])


def rel(a, b):
    return oracle.rel_l2(a, b)
