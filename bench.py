#!/usr/bin/env python3
"""Benchmark of the SSD hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step = one ssd_scan_fwd over the Mamba-2-2.7B-shaped long-context prefill
layer (batch 1, seqlen 65536, 80 heads, headdim 64, d_state 128, one group,
bf16 x/B/C, fp32 dt/A/D and states): every row of the hot path -- chunk
cumsum and decays, C.B^T, the decay mask, the intra-chunk product, chunk
states, inter-chunk state passing, the off-diagonal output and the D skip.
This is the largest prefill workload that fits one GPU.  The line also
carries the other prefill workloads (fp32 256-token, 130M 4096-token, 370M
batch-8 2048-token with a random initial state), each with its own roofline,
the decode state update (64-layer 2.7B-shaped stack at batch 1/16/64/256,
fp32 and bf16 states, single- and multi-token), cached decode against
recompute, a packed batch and the fused layer steps.

Inputs are seeded synthetic data generated on the device; the long layer's
inputs (1.4 GB) are larger than the L2 cache, and the smaller workloads
rotate through enough input/output sets to exceed twice the L2 cache, so no
step reads another step's data from L2.

--impl reference times the fp64 CPU oracle (the only other program that
computes this path here) on the host cores, on a bounded sample of the same
workload (whole heads of the layer: every head is an independent
recurrence), and prints the same line with "impl": "reference".

Under torchrun the layer's heads are split across the ranks (whole groups,
or a single group split on head-pair boundaries; B and C are inputs every
rank reads), each rank scanning its heads on its own GPU with no collective
in the data path: strong scaling, value = the layer's tokens / max over ranks
of the timed region.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "mamba2_2p7b_L65536"
EXTRA_SCANS = ("ssd_fp32_L256_H4_P64_N64", "mamba2_130m_L4096", "mamba2_370m_b8_L2048")
METRIC = "SSD prefill Mtokens/s & decode state-update GB/s, % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers
def ncu_traffic(kernel, workload, key="bytes_per_launch"):
    """DRAM bytes per launch of `kernel` on `workload` from one ncu capture
    (dram__bytes_read.sum + dram__bytes_write.sum), as recorded in
    profiles/dram_traffic.json with the hash of the kernel's sources at capture
    time; None when there is no capture or the sources have changed since."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            entry = json.load(f)[kernel][workload]
        h = hashlib.sha256()
        for src in entry["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
    except (OSError, ValueError, KeyError, TypeError):
        return None
    return entry[key] if h.hexdigest() == entry["sources_sha256"] else None


def ncu_call_traffic(workload):
    """DRAM bytes of one whole call (every kernel it launches) on `workload`
    from one ncu capture, as recorded under "calls" in
    profiles/dram_traffic.json; None when absent or the sources have changed."""
    return ncu_traffic("calls", workload, key="bytes_per_call")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = d.get("hbm_gbs") or d.get("hbm_GBs") or d.get("copy_gbs")
        tf = d.get("bf16_tflops")
        tfs = d.get("bf16_tflops_sustained", tf)
        if hbm and tf:
            return {"hbm_gbs": float(hbm), "bf16_tflops": float(tf),
                    "bf16_tflops_sustained": float(tfs), "source": "measured"}
    except (OSError, ValueError):
        pass
    out = dict(FALLBACK_PEAKS)
    out["source"] = "fallback"
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        import tempfile
        self.index = index
        self.proc = None
        # the raw samples go to SSD_CLOCKS_CSV_DIR when set (to keep them),
        # else to a temporary file; the JSON line carries their summary
        out_dir = os.environ.get("SSD_CLOCKS_CSV_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"ssd_clocks_rank{index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------- workloads
def scan_flops_bytes(shape, with_init):
    """Algorithmic work of one scan: causal-triangle FLOPs (C.B^T once per
    group) and compulsory bytes (inputs read once, outputs written once)."""
    b, L, H, P, N, G, Q = (shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                           shape.dstate, shape.ngroups, shape.chunk)
    nc = L // Q
    per_chunk = G * Q * (Q + 1) * N + H * (Q * (Q + 1) * P + 4 * Q * N * P + 2 * N * P)
    flops = b * nc * per_chunk
    es = {"bf16": 2, "fp8": 1}.get(shape.dtype, 4)   # bytes of an x, B or C value
    ey = 4 if shape.dtype == "f32" else 2            # y: bf16 for bf16 and fp8 inputs
    byts = (b * L * H * P * (es + ey)       # x read, y written
            + b * L * H * 4                 # dt
            + 2 * b * L * G * N * es        # B, C
            + 2 * H * 4                     # A, D
            + b * H * P * N * 4 * (2 if with_init else 1))  # init (if any), final
    return flops, byts


def make_scan_set(shape, seed, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    b, L, H, P, N, G = (shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                        shape.dstate, shape.ngroups)
    dt_ = {"bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn}.get(shape.dtype, torch.float32)
    lo, hi = -6.907755278982137, -2.3025850929940455
    t = {
        "x": torch.randn((b, L, H, P), generator=g, device=device).to(dt_),
        "dt": torch.exp(lo + (hi - lo) * torch.rand((b, L, H), generator=g, device=device)),
        "A": -torch.exp(2.772588722239781 * torch.rand((H,), generator=g, device=device)),
        "B": torch.randn((b, L, G, N), generator=g, device=device).to(dt_),
        "C": torch.randn((b, L, G, N), generator=g, device=device).to(dt_),
        "D": torch.randn((H,), generator=g, device=device),
        "init": (0.1 * torch.randn((b, H, P, N), generator=g, device=device)
                 if shape.random_init else None),
    }
    t["y"] = torch.empty(t["x"].shape, dtype=torch.bfloat16 if shape.dtype == "fp8" else dt_,
                         device=device)
    t["final"] = torch.empty((b, H, P, N), dtype=torch.float32, device=device)
    return t


def torch_input_dtype(shape):
    import torch
    return {"bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn}.get(shape.dtype, torch.float32)


def time_scan(shape, steps, warmup, device, l2_bytes, dist=None, graph=True):
    """Times `steps` consecutive ssd_scan_fwd calls, each on its own rotating
    input/output set.  With graph=True the K calls are captured into a CUDA
    graph (after `warmup` eager calls and one untimed replay) and the timed
    region is one replay, so host-side call overhead is not measured.  A
    second, separately timed graph records CUDA events around each call's
    y-writing kernel (the library's profiling hook) to time that kernel alone;
    it is kept apart because the extra event records serialise the kernels the
    library otherwise lets overlap.
    Returns (ms per call, ms of the y-writing kernel per call, sets, bytes)."""
    import torch
    import state_space_model_chunked_gb300 as ssd
    _, byts = scan_flops_bytes(shape, shape.random_init)
    nsets = max(1, -(-2 * l2_bytes // max(byts, 1)))
    sets = [make_scan_set(shape, 1000 + i, device) for i in range(nsets)]
    ws_bytes = ssd.scan_workspace_bytes(shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                                        shape.dstate, shape.ngroups, shape.chunk,
                                        dtype=torch_input_dtype(shape), device=device)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)

    def step(i):
        s = sets[i % nsets]
        ssd.scan_fwd(s["x"], s["dt"], s["A"], s["B"], s["C"], s["D"], shape.chunk, s["init"],
                     y=s["y"], final_state=s["final"], workspace=ws)

    for i in range(warmup):
        step(i)
    stream = torch.cuda.current_stream(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(device)

    def run(profile):
        if profile:
            for i in range(steps):
                ssd.scan_profile_events(*ev[i])
                step(warmup + i)
            ssd.scan_profile_events(None, None)
        else:
            for i in range(steps):
                step(warmup + i)

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(device)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        if dist is not None:
            dist.barrier()
        return e0.elapsed_time(e1)

    if graph:
        graphs = {}
        for prof in (False, True):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                run(prof)
            g.replay()                                   # untimed
            torch.cuda.synchronize(device)
            graphs[prof] = g
        ms = timed(graphs[False].replay) / steps
        timed(graphs[True].replay)
    else:
        ms = timed(lambda: run(False)) / steps
        timed(lambda: run(True))
    kern_ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    return ms, kern_ms, nsets, byts


def time_scan_e2e(shape, steps, warmup, device):
    """Mtokens/s through the public API with pinned host buffers: per step the
    host->device copy of the inputs, the scan, and the device->host copy of y
    and the final state, with consecutive steps overlapped by the library's
    HostScanPipeline (one step's inputs in flight while the previous one
    computes and the one before returns its outputs).  Host wall time from the
    first copy of the first timed step to the last byte of the last one."""
    import torch
    import state_space_model_chunked_gb300 as ssd
    s = make_scan_set(shape, 77, device)
    host = {k: (v.cpu().pin_memory() if v is not None else None)
            for k, v in s.items() if k not in ("y", "final")}
    pipe = ssd.HostScanPipeline(device)
    outs = [(torch.empty(s["y"].shape, dtype=s["y"].dtype, pin_memory=True),
             torch.empty(s["final"].shape, dtype=torch.float32, pin_memory=True))
            for _ in range(pipe.depth)]
    out = outs[0]

    def step(i):
        pipe.submit(host["x"], host["dt"], host["A"], host["B"], host["C"], host["D"],
                    shape.chunk, host["init"], out=outs[i % pipe.depth])

    for i in range(max(warmup, 1)):
        step(i)
    pipe.synchronize()
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    pipe.synchronize()
    dt = (time.perf_counter() - t0) / steps
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = out[0].numel() * out[0].element_size() + out[1].numel() * 4
    return dt, h2d, d2h


def time_decode(batch, steps, device, peaks, state_dtype=None):
    """One ssd_state_update per token over the 64-layer 2.7B-shaped stack,
    layers flattened into heads (one group per layer); the state in fp32, or
    stored as bf16 with state_dtype=torch.bfloat16."""
    import torch
    import state_space_model_chunked_gb300 as ssd
    from state_space_model_chunked_gb300 import inputs as gen
    ds = gen.DECODE_SHAPE
    Hf, G, P, N = ds.layers * ds.nheads, ds.layers, ds.headdim, ds.dstate
    state = gen.device_decode_state(batch, Hf, P, N, seed=batch, device=device)
    if state_dtype is not None and state_dtype != state.dtype:
        state = state.to(state_dtype)
    A, D = gen.decode_params(Hf, seed=batch)
    A, D = torch.from_numpy(A).to(device), torch.from_numpy(D).to(device)
    ntok = 4
    toks = [gen.device_decode_token_inputs(batch, Hf, P, N, G, seed=batch, step=i, device=device)
            for i in range(ntok)]
    y = torch.empty((batch, Hf, P), dtype=torch.bfloat16, device=device)
    for i in range(3):
        t = toks[i % ntok]
        ssd.state_update(state, t["x"], t["dt"], A, t["B"], t["C"], D, y=y)
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for i in range(steps):
        t = toks[i % ntok]
        ssd.state_update(state, t["x"], t["dt"], A, t["B"], t["C"], D, y=y)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    byts = (2 * batch * Hf * P * N * state.element_size() + 2 * batch * Hf * P * 2
            + batch * Hf * 4 + 2 * batch * G * N * 2 + 2 * Hf * 4)
    gbs = byts / (ms * 1e-3) / 1e9
    sdt = str(state.dtype).replace("torch.", "")
    del state, toks
    torch.cuda.empty_cache()
    return {"batch": batch, "state": sdt, "steps": steps, "ms_per_step": ms,
            "bytes_per_step": byts,
            "GB_per_s": gbs, "frac_of_measured_hbm": gbs / peaks["hbm_gbs"],
            "frac_of_8TBs_nominal": gbs / 8000.0}


def time_decode_multi(batch, ntok, steps, device, peaks):
    """The 64-layer 2.7B-shaped decode stack (layers flattened into heads, one
    group per layer) advanced `ntok` tokens per ssd_state_update_multi call:
    each state is read and written once per call.  Tokens/s counts batch x
    ntok tokens through the whole stack per call."""
    import torch
    import state_space_model_chunked_gb300 as ssd
    from state_space_model_chunked_gb300 import inputs as gen
    ds = gen.DECODE_SHAPE
    Hf, G, P, N = ds.layers * ds.nheads, ds.layers, ds.headdim, ds.dstate
    state = gen.device_decode_state(batch, Hf, P, N, seed=batch, device=device)
    A, D = gen.decode_params(Hf, seed=batch)
    A, D = torch.from_numpy(A).to(device), torch.from_numpy(D).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(1000 + ntok)
    x = torch.randn((batch, ntok, Hf, P), generator=g, device=device).to(torch.bfloat16)
    dt = torch.exp(gen.LN_DT_LO + (gen.LN_DT_HI - gen.LN_DT_LO)
                   * torch.rand((batch, ntok, Hf), generator=g, device=device))
    B = torch.randn((batch, ntok, G, N), generator=g, device=device).to(torch.bfloat16)
    C = torch.randn((batch, ntok, G, N), generator=g, device=device).to(torch.bfloat16)
    y = torch.empty_like(x)
    for _ in range(3):
        ssd.state_update_multi(state, x, dt, A, B, C, D, y=y)
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(steps):
        ssd.state_update_multi(state, x, dt, A, B, C, D, y=y)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    byts = (2 * batch * Hf * P * N * 4
            + ntok * (2 * batch * Hf * P * 2 + batch * Hf * 4 + 2 * batch * G * N * 2)
            + 2 * Hf * 4)
    gbs = byts / (ms * 1e-3) / 1e9
    del state, x, dt, B, C, y
    torch.cuda.empty_cache()
    return {"batch": batch, "tokens_per_call": ntok, "ms_per_call": ms,
            "ms_per_token": ms / ntok,
            "tokens_per_s": batch * ntok / (ms * 1e-3),
            "bytes_per_call": byts, "GB_per_s": gbs,
            "frac_of_measured_hbm": gbs / peaks["hbm_gbs"]}


def time_decode_per_layer(batch, steps, device, peaks):
    """The same decode stack as 64 per-layer ssd_state_update calls per token
    (each layer's state, x, B, C contiguous; 80 heads, one group), the 64 calls
    of one token captured in a CUDA graph; four tokens' inputs rotate."""
    import torch
    import state_space_model_chunked_gb300 as ssd
    from state_space_model_chunked_gb300 import inputs as gen
    ds = gen.DECODE_SHAPE
    nl, H, P, N = ds.layers, ds.nheads, ds.headdim, ds.dstate
    states = [gen.device_decode_state(batch, H, P, N, seed=batch * 100 + l, device=device)
              for l in range(nl)]
    A, D = gen.decode_params(nl * H, seed=batch)
    A = torch.from_numpy(A).to(device).view(nl, H)
    D = torch.from_numpy(D).to(device).view(nl, H)
    ntok = 4
    toks = [[gen.device_decode_token_inputs(batch, H, P, N, 1, seed=batch * 100 + l, step=i,
                                            device=device) for l in range(nl)]
            for i in range(ntok)]
    ys = [torch.empty((batch, H, P), dtype=torch.bfloat16, device=device) for _ in range(nl)]

    def token(i):
        for l in range(nl):
            t = toks[i][l]
            ssd.state_update(states[l], t["x"], t["dt"], A[l], t["B"], t["C"], D[l], y=ys[l])

    stream = torch.cuda.Stream(device)
    graphs = []
    with torch.cuda.stream(stream):
        for i in range(ntok):
            token(i)                      # warm-up outside capture
        torch.cuda.synchronize(device)
        for i in range(ntok):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                token(i)
            graphs.append(g)
        for i in range(3):
            graphs[i % ntok].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record(stream)
        for i in range(steps):
            graphs[i % ntok].replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    Hf, G = nl * H, nl
    byts = (2 * batch * Hf * P * N * 4 + 2 * batch * Hf * P * 2 + batch * Hf * 4
            + 2 * batch * G * N * 2 + 2 * Hf * 4)
    gbs = byts / (ms * 1e-3) / 1e9
    del states, toks, graphs
    torch.cuda.empty_cache()
    return {"batch": batch, "steps": steps, "launch": "64 per-layer calls per token in a CUDA graph",
            "ms_per_step": ms, "GB_per_s": gbs, "frac_of_measured_hbm": gbs / peaks["hbm_gbs"]}


def time_decode_vs_recompute(device, prefixes=(4096, 65536), reps=20):
    """One 2.7B-shaped layer (80 heads, headdim 64, d_state 128), batch 1: the
    next token's output from the cached state (one ssd_state_update) against
    recomputing it from scratch (ssd_scan_fwd over the prefix plus the token)."""
    import torch
    import state_space_model_chunked_gb300 as ssd
    from state_space_model_chunked_gb300 import inputs as gen
    H, P, N = 80, 64, 128
    out = []
    A, D = gen.decode_params(H, seed=3)
    A, D = torch.from_numpy(A).to(device), torch.from_numpy(D).to(device)
    state = gen.device_decode_state(1, H, P, N, seed=3, device=device)
    tok = gen.device_decode_token_inputs(1, H, P, N, 1, seed=3, step=0, device=device)
    stream = torch.cuda.current_stream(device)

    def timed(fn):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps

    dec_ms = timed(lambda: ssd.state_update(state, tok["x"], tok["dt"], A, tok["B"], tok["C"], D))
    for T in prefixes:
        g = torch.Generator(device=device)
        g.manual_seed(T)
        L = T + 1
        x = torch.randn((1, L, H, P), generator=g, device=device).to(torch.bfloat16)
        dt = torch.exp(-6.9 + 4.6 * torch.rand((1, L, H), generator=g, device=device))
        B = torch.randn((1, L, 1, N), generator=g, device=device).to(torch.bfloat16)
        C = torch.randn((1, L, 1, N), generator=g, device=device).to(torch.bfloat16)
        ws = torch.empty(max(ssd.scan_workspace_bytes(1, L, H, P, N, 1, 256, device=device), 1),
                         dtype=torch.uint8, device=device)
        y = torch.empty_like(x)
        fin = torch.empty((1, H, P, N), dtype=torch.float32, device=device)
        scan_ms = timed(lambda: ssd.scan_fwd(x, dt, A, B, C, D, 256, None, y=y, final_state=fin,
                                             workspace=ws))
        out.append({"prefix_tokens": T, "recompute_ms": scan_ms, "cached_decode_ms": dec_ms,
                    "speedup": scan_ms / dec_ms})
        del x, dt, B, C, ws, y
    torch.cuda.empty_cache()
    return out


def time_varlen(device, peaks, total=65536, reps=10):
    """A packed batch of the 80-head layer (headdim 64, d_state 128): sequences
    of log-uniform lengths in [64, 8192] tokens, `total` tokens in all, as one
    ssd_scan_fwd_varlen call, against the batched call on the same sequences
    each padded to the longest (what the batched entry point needs)."""
    import numpy as np
    import torch
    import state_space_model_chunked_gb300 as ssd
    from state_space_model_chunked_gb300 import inputs as gen
    H, P, N = 80, 64, 128
    lengths, acc = [], 0
    for v in gen.packed_lengths(256, 64, 8192, seed=5):
        v = min(v, total - acc)
        lengths.append(v)
        acc += v
        if acc == total:
            break
    nseq, Lmax = len(lengths), max(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    g = torch.Generator(device=device)
    g.manual_seed(77)

    def tensors(shape_x, shape_dt, shape_bc):
        return (torch.randn(shape_x, generator=g, device=device).to(torch.bfloat16),
                torch.exp(-6.9 + 4.6 * torch.rand(shape_dt, generator=g, device=device)),
                torch.randn(shape_bc, generator=g, device=device).to(torch.bfloat16),
                torch.randn(shape_bc, generator=g, device=device).to(torch.bfloat16))

    A = -torch.exp(2.77 * torch.rand((H,), generator=g, device=device))
    D = torch.randn((H,), generator=g, device=device)
    stream = torch.cuda.current_stream(device)

    def timed(fn):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps

    x, dt, B, C = tensors((total, H, P), (total, H), (total, 1, N))
    y = torch.empty_like(x)
    fin = torch.empty((nseq, H, P, N), dtype=torch.float32, device=device)
    cu_dev = torch.from_numpy(cu).to(device)
    ws = torch.empty(max(ssd.scan_varlen_workspace_bytes(cu, H, P, N, 1, 256, device=device), 1),
                     dtype=torch.uint8, device=device)
    packed_ms = timed(lambda: ssd.scan_fwd_varlen(x, dt, A, B, C, cu, D, 256, None, y=y,
                                                  final_state=fin, workspace=ws,
                                                  cu_seqlens_dev=cu_dev))
    byts = 2 * total * H * P * 2 + total * H * 4 + 2 * total * N * 2 + nseq * H * P * N * 4
    del x, dt, B, C, y, ws
    xp, dtp, Bp, Cp = tensors((nseq, Lmax, H, P), (nseq, Lmax, H), (nseq, Lmax, 1, N))
    yp = torch.empty_like(xp)
    finp = torch.empty((nseq, H, P, N), dtype=torch.float32, device=device)
    wsp = torch.empty(max(ssd.scan_workspace_bytes(nseq, Lmax, H, P, N, 1, 256, device=device),
                          1), dtype=torch.uint8, device=device)
    padded_ms = timed(lambda: ssd.scan_fwd(xp, dtp, A, Bp, Cp, D, 256, None, y=yp,
                                           final_state=finp, workspace=wsp))
    del xp, dtp, Bp, Cp, yp, wsp
    torch.cuda.empty_cache()
    achieved = byts / (packed_ms * 1e-3) / 1e9
    return {"workload": f"mamba2_2p7b packed: {nseq} sequences, log-uniform lengths "
                        f"64..8192, {total} tokens (longest {Lmax})",
            "packed_ms": packed_ms, "packed_Mtokens_per_s": total / (packed_ms * 1e-3) / 1e6,
            "padded_ms": padded_ms, "padded_Mtokens_per_s": total / (padded_ms * 1e-3) / 1e6,
            "call_roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                              "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"]}}


def time_fused_steps(shape, device, reps=20):
    """The workload's scan with the layer's neighbouring steps fused (dt bias +
    softplus + clamp on the input side, the silu(z) gate on the output side)
    against the plain scan, on rotating input sets larger than L2."""
    import torch
    import state_space_model_chunked_gb300 as ssd
    nsets = 10
    sets = [make_scan_set(shape, 2000 + i, device) for i in range(nsets)]
    g = torch.Generator(device=device)
    g.manual_seed(5)
    for s in sets:
        s["z"] = torch.randn(s["x"].shape, generator=g, device=device).to(s["x"].dtype)
    bias = torch.randn((shape.nheads,), generator=g, device=device) * 0.5
    ws = torch.empty(max(ssd.scan_workspace_bytes(shape.batch, shape.seqlen, shape.nheads,
                                                  shape.headdim, shape.dstate, shape.ngroups,
                                                  shape.chunk, device=device,
                                                  dt_transform=True), 1),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def timed(dt_on, gate_on):
        def call(i):
            s = sets[i % nsets]
            extra = {}
            if dt_on:
                extra.update(dt_bias=bias, dt_softplus=True, dt_limit=(1e-4, 0.1))
            if gate_on:
                extra["z"] = s["z"]
            ssd.scan_fwd(s["x"], s["dt"], s["A"], s["B"], s["C"], s["D"], shape.chunk,
                         s["init"], y=s["y"], final_state=s["final"], workspace=ws, **extra)
        for i in range(3):
            call(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record(stream)
        for i in range(reps):
            call(i)
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps

    plain, dt_only, gate_only, fused = (timed(False, False), timed(True, False),
                                        timed(False, True), timed(True, True))
    del sets, ws
    torch.cuda.empty_cache()
    return {"workload": shape.name, "plain_ms": plain, "dt_transform_ms": dt_only,
            "gate_ms": gate_only, "fused_ms": fused,
            "fused_extra_bytes": shape.batch * shape.seqlen * shape.nheads * shape.headdim * 2,
            "note": "eager calls (host overhead included in both)"}


def time_fp8_inputs(device, peaks, l2, bf16_ms, steps=20):
    """The long-context layer with 8-bit E4M3 x, B, C: the whole call (the
    widening of x, B, C to bfloat16 copies, then the bf16 path), and the
    widening kernel alone on as many values, timed with CUDA events on its
    stream (1 byte read and 2 written per value: its HBM roofline)."""
    import torch
    import state_space_model_chunked_gb300 as ssd
    from state_space_model_chunked_gb300 import inputs as gen
    sh = gen.SCAN_SHAPES["mamba2_2p7b_L65536_fp8"]
    ms, kern_ms, _, byts = time_scan(sh, steps, 5, device, l2)
    entry = scan_line_entry(sh, ms, kern_ms, byts, peaks, "ssd_tc_scan_kernel")
    torch.cuda.empty_cache()
    n = sh.batch * sh.seqlen * (sh.nheads * sh.headdim + 2 * sh.ngroups * sh.dstate)
    g = torch.Generator(device=device)
    g.manual_seed(3)
    nbuf = 2                                  # 0.35 GB in, 0.7 GB out each: beyond L2
    src = [torch.randn(n, generator=g, device=device).to(torch.float8_e4m3fn)
           for _ in range(nbuf)]
    dst = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(nbuf)]
    for i in range(3):
        ssd.fp8_e4m3_to_bf16(src[i % nbuf], out=dst[i % nbuf])
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for i in range(steps):
        ssd.fp8_e4m3_to_bf16(src[i % nbuf], out=dst[i % nbuf])
    e1.record(stream)
    torch.cuda.synchronize(device)
    wms = e0.elapsed_time(e1) / steps
    del src, dst
    torch.cuda.empty_cache()
    achieved = 3 * n / (wms * 1e-3) / 1e9
    entry["roofline"]["call_traffic"] = ncu_call_traffic(sh.name)
    entry.update({
        "inputs": "x, B, C as float8_e4m3fn; y bfloat16",
        "vs_bf16_inputs": bf16_ms / ms,
        "widen": {"kernel": "ssd_fp8_widen_kernel", "values": n, "ms": wms, "bound": "hbm",
                  "algorithmic_bytes": 3 * n, "achieved": achieved, "peak": peaks["hbm_gbs"],
                  "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                  "traffic": ncu_traffic("ssd_fp8_widen_kernel", sh.name)},
    })
    return entry


def time_gated_norm_pass(shape, device, reps=20):
    """Cost of the step the scan kernels do not fuse: the gated RMS norm over
    all heads of a token (y * silu(z), then x / rms(x) * w over nheads x
    headdim), as a separate pass with torch ops on the layer's y and z.  It
    reads y and z and writes the result: 3 bytes moved per output byte."""
    import torch
    import torch.nn.functional as F
    b, L, H, P = shape.batch, shape.seqlen, shape.nheads, shape.headdim
    g = torch.Generator(device=device)
    g.manual_seed(9)
    y = torch.randn((b, L, H * P), generator=g, device=device).to(torch.bfloat16)
    z = torch.randn((b, L, H * P), generator=g, device=device).to(torch.bfloat16)
    w = torch.ones((H * P,), device=device, dtype=torch.bfloat16)
    out = torch.empty_like(y)

    def one():
        out.copy_(F.rms_norm(y * F.silu(z), (H * P,), w, eps=1e-5))

    for _ in range(3):
        one()
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(reps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / reps
    byts = 3 * y.numel() * 2
    del y, z, out
    torch.cuda.empty_cache()
    return {"workload": shape.name, "ms": ms, "compulsory_bytes": byts,
            "roofline_ms": byts / 6.79e12 * 1e3,
            "note": "torch ops (not this library): the unfused gated normalisation after the scan"}


def cpu_oracle_sample(shape, heads=None, target_s=10.0, cores=None, max_reps=50):
    """The oracle as it stands on the host cores, on `heads` whole heads of the
    workload (all of them by default; every head is an independent
    recurrence), repeated until `target_s` seconds have passed.  The inputs
    are drawn before the clock starts.  Returns (Mtokens/s of the whole layer,
    cores used, sample description)."""
    import oracle
    from state_space_model_chunked_gb300 import inputs as gen
    cores = cores or os.cpu_count() or 1
    heads = heads or shape.nheads
    inp = gen.scan_inputs(shape.batch, shape.seqlen, heads, shape.headdim, shape.dstate,
                          min(shape.ngroups, heads), shape.dtype, seed=5,
                          random_init=shape.random_init)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                        inp["init"], nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s or reps >= max_reps:
            break
    tok_s = reps * shape.tokens * heads / shape.nheads / el
    desc = (f"{reps} pass(es) of {heads} of the {shape.nheads} heads of {shape.name} "
            f"({shape.tokens} tokens) through the fp64 oracle on {cores} thread(s), "
            f"{el:.1f} s, scaled to the whole layer")
    return tok_s / 1e6, cores, desc


def executed_tc_flops(shape):
    """FLOPs the tensor-core scan kernel issues on tcgen05 for one call: per
    128-token tile and head pair C.B^T, the state update, the off-diagonal
    product and both heads' masked products, each 2 x 128^3 (a single head
    per CTA: C.B^T plus three 128 x 64 x 128 products)."""
    tiles = -(-shape.seqlen // 128)
    per_group = shape.nheads // shape.ngroups
    unit = 2 * 128 ** 3
    if per_group % 2 == 0:
        return shape.batch * tiles * (shape.nheads // 2) * 4 * unit
    return shape.batch * tiles * shape.nheads * 2.5 * unit


def scan_line_entry(shape, ms, kern_ms, byts, peaks, kernel):
    """Throughput and roofline of one prefill workload: the y-writing
    kernel's fraction (compulsory bytes / its time) and the call's (the same
    bytes / the whole call's time, all its kernels)."""
    flops, _ = scan_flops_bytes(shape, shape.random_init)
    achieved = byts / (kern_ms * 1e-3) / 1e9
    call = byts / (ms * 1e-3) / 1e9
    return {
        "workload": shape.name, "ms_per_step": ms,
        "Mtokens_per_s": shape.tokens / (ms * 1e-3) / 1e6,
        "roofline": {"bound": "hbm", "kernel": kernel, "kernel_ms": kern_ms,
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "call_achieved": call,
                     "call_frac": call / peaks["hbm_gbs"], "algorithmic_bytes": byts,
                     "algorithmic_tflops": flops / (ms * 1e-3) / 1e12},
    }


def sharded_shape(shape, world, rank):
    """The rank's part of the layer: its heads (and the groups they read)."""
    import dataclasses
    from state_space_model_chunked_gb300.sharding import head_shard
    h0, h1, g0, g1 = head_shard(shape.nheads, shape.ngroups, world, rank)
    return dataclasses.replace(shape, nheads=max(h1 - h0, 0), ngroups=max(g1 - g0, 1)), (h0, h1)


# ------------------------------------------------------------------ arms
def workload_config(shape):
    """The line's `config`: the workload, identical in both arms."""
    return {"workload": shape.name, "batch": shape.batch, "seqlen": shape.seqlen,
            "nheads": shape.nheads, "headdim": shape.headdim, "dstate": shape.dstate,
            "ngroups": shape.ngroups, "chunk": shape.chunk,
            "l2": "inputs and outputs of a step (1.4 GB) larger than L2"}


def run_reference(args):
    """The oracle as it stands, timed on the host cores: each step is one pass
    over a sample of whole heads of the layer (inputs drawn before timing)."""
    import numpy as np  # noqa: F401
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    from state_space_model_chunked_gb300 import inputs as gen
    import oracle
    oracle.build()
    shape = gen.SCAN_SHAPES[WORKLOAD]
    heads = args.reference_heads
    cores = os.cpu_count() or 1
    inp = gen.scan_inputs(shape.batch, shape.seqlen, heads, shape.headdim, shape.dstate,
                          min(shape.ngroups, heads), shape.dtype, seed=5,
                          random_init=shape.random_init)

    def one():
        oracle.scan_seq(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                        inp["init"], nthreads=cores)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    layer_tokens = shape.tokens * heads / shape.nheads      # whole-layer tokens per step
    value = args.steps * layer_tokens / el / 1e6
    sample = (f"each step: {heads} of the {shape.nheads} heads of {WORKLOAD} "
              f"({shape.tokens} tokens each), scaled to the whole layer; inputs drawn before timing")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Mtokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "strong" if world > 1 else "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded PCG64)",
        "config": workload_config(shape),
        "cpu_baseline": {"value": value, "unit": "Mtokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "Mtokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_only(args):
    """One workload alone, a few launches: used for ncu captures."""
    import torch
    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    from state_space_model_chunked_gb300 import build as ssd_build
    from state_space_model_chunked_gb300 import inputs as gen
    ssd_build.build()
    peaks = load_peaks()
    if args.only == "decode":
        r = time_decode(args.decode_batch, args.steps, device, peaks,
                        torch.bfloat16 if args.decode_state == "bf16" else None)
    elif args.only == "decode_multi":
        r = time_decode_multi(args.decode_batch, args.decode_tokens, args.steps, device, peaks)
    elif args.only == "decode_per_layer":
        r = time_decode_per_layer(args.decode_batch, args.steps, device, peaks)
    else:
        props = torch.cuda.get_device_properties(device)
        l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024) or 126 * 1024 * 1024
        name = {"long": WORKLOAD, "130m": "mamba2_130m_L4096",
                "370m": "mamba2_370m_b8_L2048", "fp8": "mamba2_2p7b_L65536_fp8"}[args.only]
        shape = gen.SCAN_SHAPES[name]
        ms, kern, _, byts = time_scan(shape, args.steps, args.warmup, device, l2, graph=False)
        r = {"workload": name, "ms_per_step": ms, "scan_kernel_ms": kern,
             "GB_per_s": byts / (ms * 1e-3) / 1e9}
    print(json.dumps({"only": args.only, **r}), flush=True)
    return 0


def run_gpu(args):
    import torch
    world, rank, local = dist_setup()
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    import state_space_model_chunked_gb300 as ssd
    from state_space_model_chunked_gb300 import build as ssd_build
    from state_space_model_chunked_gb300 import inputs as gen
    from state_space_model_chunked_gb300.sharding import max_over_ranks
    if rank == 0 or world == 1:
        ssd_build.build()
    if dist is not None:
        dist.barrier()
    ssd.load()
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024) or 126 * 1024 * 1024
    full = gen.SCAN_SHAPES[WORKLOAD]
    shape, (h0, h1) = sharded_shape(full, world, rank)
    _, full_bytes = scan_flops_bytes(full, full.random_init)

    with ClockSampler(local) as clk:
        if shape.nheads > 0:
            ms, kern_ms, nsets, byts = time_scan(shape, args.steps, args.warmup, device, l2, dist)
        else:   # more ranks than the layer splits into: this rank only joins the
            # barriers time_scan takes (two timed replays, two barriers each)
            if dist is not None:
                for _ in range(4):
                    dist.barrier()
            ms, kern_ms, nsets, byts = 0.0, 0.0, 1, 0
        ms = max_over_ranks(ms, dist, device)
        kern_ms = max_over_ranks(kern_ms, dist, device)
        extra = {}
        if world == 1 and not args.quick:
            configs = []
            for name in EXTRA_SCANS:
                sh = gen.SCAN_SHAPES[name]
                sms, skern, _, sbytes = time_scan(sh, 20, 5, device, l2)
                kname = "ssd_tc_scan_kernel" if sh.dtype == "bf16" else "ssd_scan_simt_kernel"
                configs.append(scan_line_entry(sh, sms, skern, sbytes, peaks, kname))
            extra["other_prefill_workloads"] = configs
            torch.cuda.empty_cache()
            extra["decode"] = [time_decode(b, 128, device, peaks) for b in (1, 16, 64, 256)]
            extra["decode_bf16_state"] = [time_decode(b, 128, device, peaks, torch.bfloat16)
                                          for b in (1, 16, 64, 256)]
            extra["decode_per_layer"] = [time_decode_per_layer(b, 32, device, peaks)
                                         for b in (1, 16)]
            extra["decode_multi_token"] = [time_decode_multi(b, t, 10, device, peaks)
                                           for b in (1, 16) for t in (4, 16)]
            extra["decode_vs_recompute"] = time_decode_vs_recompute(device)
            extra["varlen"] = time_varlen(device, peaks)
            extra["fused_steps"] = [time_fused_steps(gen.SCAN_SHAPES[n], device)
                                    for n in ("mamba2_130m_L4096", WORKLOAD)]
            extra["gated_norm_separate_pass"] = time_gated_norm_pass(full, device)
            extra["fp8_inputs"] = time_fp8_inputs(device, peaks, l2, ms)
    clocks = clk.summary()

    # the same K steps as the device-timed region, back to back through the
    # pipeline (its fill and drain, one unpaired copy each way, included once)
    e2e_s, h2d, d2h = ((time_scan_e2e(shape, max(args.steps, 3), args.warmup, device))
                       if shape.nheads > 0 else (0.0, 0, 0))
    e2e_s = max_over_ranks(e2e_s, dist, device)
    h2d = int(max_over_ranks(h2d, dist, device)) * world
    d2h = int(max_over_ranks(d2h, dist, device)) * world
    value = full.tokens / (ms * 1e-3) / 1e6
    entry = scan_line_entry(full, ms, kern_ms, full_bytes, peaks, "ssd_tc_scan_kernel")
    roof = dict(entry["roofline"])
    roof.update({"peak_source": peaks["source"],
                 "traffic": ncu_traffic("ssd_tc_scan_kernel", WORKLOAD),
                 "call_traffic": ncu_call_traffic(WORKLOAD)})
    if world == 1:
        tflops = executed_tc_flops(full) / (kern_ms * 1e-3) / 1e12
        roof["tensor"] = {"executed_tflops": tflops, "peak_tflops": peaks["bf16_tflops"],
                          "frac": tflops / peaks["bf16_tflops"],
                          "note": "tcgen05 FLOPs the scan kernel issues (full 128-token "
                                  "tiles) / its time"}
    launches = (ssd.scan_kernel_launches(shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                                         shape.dstate, shape.ngroups, shape.chunk, device=device)
                if shape.nheads > 0 else 0)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "Mtokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong" if world > 1 else "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, generated on device)",
        "config": workload_config(full),
        "timing": {"launch": "K calls captured in one CUDA graph, timed as one replay",
                   "inputs": (f"one set per rank ({byts / 1e6:.0f} MB, larger than L2)"
                              if nsets == 1 else f"rotating {nsets} input/output sets "
                                                 f"({nsets * byts / 1e6:.0f} MB > 2x L2)"),
                   "parallelism": (f"heads split over {world} GPUs ({shape.nheads} each)"
                                   if world > 1 else "one GPU")},
        "roofline": roof,
        "e2e": {"value": full.tokens / e2e_s / 1e6, "unit": "Mtokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "HostScanPipeline: pinned host inputs copied in, the scan, y and the "
                       "final state copied out, consecutive steps overlapped",
                "steps": max(args.steps, 3)},
        "gpu_launches": launches * args.steps * world,
        "clocks": clocks,
    }
    line.update(extra)
    if not args.no_cpu and world == 1:
        v, cores, desc = cpu_oracle_sample(full, target_s=args.cpu_seconds)
        v1, _, desc1 = cpu_oracle_sample(full, heads=4, target_s=0.0, cores=1, max_reps=1)
        line["cpu_baseline"] = {"value": v, "unit": "Mtokens/s", "cores": cores,
                                "kind": "oracle", "sample": desc,
                                "one_core": {"value": v1, "unit": "Mtokens/s", "cores": 1,
                                             "sample": desc1}}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--only", choices=["decode", "decode_multi", "decode_per_layer", "long", "130m",
                                       "370m", "fp8"],
                    default=None, help="run one workload alone (for profiler captures)")
    ap.add_argument("--decode-batch", type=int, default=16)
    ap.add_argument("--decode-tokens", type=int, default=16,
                    help="tokens per call of the --only decode_multi run")
    ap.add_argument("--reference-heads", type=int, default=16,
                    help="heads of the layer per step of the reference arm")
    ap.add_argument("--decode-state", choices=["f32", "bf16"], default="f32",
                    help="state storage of the --only decode run")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.only:
        return run_only(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
