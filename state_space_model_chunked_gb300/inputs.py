"""Seeded synthetic inputs for the SSD scan and decode workloads.

This module serves both the CUDA path and the fp64 oracle and holds none of
the method's arithmetic: it only draws random numbers and encodes them.

Distributions (the same for every workload):
  x, B, C ~ N(0, 1), rounded to bfloat16 (round-to-nearest-even) when the
          workload's input dtype is bf16, encoded as 8-bit E4M3 codes
          (nearest-even, torch's float8_e4m3fn cast) when it is fp8;
  dt      = exp(U(ln 1e-3, ln 1e-1)), one value per (batch, token, head);
  A_h     = -exp(U(0, ln 16)), one value per head;
  D_h     ~ N(0, 1);
  init    = zeros, or N(0, 0.1^2) where the workload asks for a random one;
  decode states ~ N(0, 1).

Host generation uses numpy's PCG64; the decode workloads whose state would not
fit on the host draw on the device with a seeded torch generator instead (see
``device_decode_state``).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

LN_DT_LO = float(np.log(1e-3))
LN_DT_HI = float(np.log(1e-1))
LN_A_HI = float(np.log(16.0))


@dataclass(frozen=True)
class ScanShape:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str            # "f32", "bf16" or "fp8": dtype of x, B, C (y is bf16 for fp8)
    random_init: bool = False

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


@dataclass(frozen=True)
class DecodeShape:
    name: str
    layers: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    batches: tuple = field(default=(1, 16, 64, 256))
    steps: int = 128
    dtype: str = "bf16"


# The workloads, named by what they are.
SCAN_SHAPES = {
    "ssd_fp32_L256_H4_P64_N64": ScanShape("ssd_fp32_L256_H4_P64_N64", 1, 256, 4, 64, 64, 1, 64, "f32"),
    "mamba2_130m_L4096": ScanShape("mamba2_130m_L4096", 1, 4096, 24, 64, 128, 1, 256, "bf16"),
    "mamba2_370m_b8_L2048": ScanShape("mamba2_370m_b8_L2048", 8, 2048, 32, 64, 128, 1, 256, "bf16", True),
    "mamba2_2p7b_L65536": ScanShape("mamba2_2p7b_L65536", 1, 65536, 80, 64, 128, 1, 256, "bf16"),
    # the same layer with 8-bit E4M3 x, B, C (bf16 y)
    "mamba2_2p7b_L65536_fp8": ScanShape("mamba2_2p7b_L65536_fp8", 1, 65536, 80, 64, 128, 1, 256,
                                        "fp8"),
}
DECODE_SHAPE = DecodeShape("mamba2_2p7b_decode_64layers", 64, 80, 64, 128, 1)


def bf16_round(a):
    """Round float32 values to bfloat16 (nearest-even).  Returns (values as
    float32, raw uint16 bit patterns)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    bits = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    vals = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return vals, bits


def e4m3_encode(a):
    """float32 values -> 8-bit E4M3 codes (uint8), rounded to nearest even by
    torch's float8_e4m3fn cast on the host.  Values must lie within +-448."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def _normal(rng, shape, dtype):
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == "bf16":
        v, _ = bf16_round(v)
    elif dtype == "fp8":
        return e4m3_encode(v)
    return v


def scan_inputs(batch, seqlen, nheads, headdim, dstate, ngroups, dtype="bf16",
                seed=0, random_init=False, with_D=True):
    """Inputs for one scan.  Every array is float32 holding exactly the values
    the GPU sees (bf16-representable where dtype == 'bf16'), except that for
    dtype == 'fp8' x, B and C are uint8 arrays of E4M3 codes.

    Returns dict with x [b,L,H,P], dt [b,L,H], A [H], B, C [b,L,G,N],
    D [H] (or None), init [b,H,P,N] (or None)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    out["x"] = _normal(rng, (batch, seqlen, nheads, headdim), dtype)
    out["dt"] = np.exp(rng.uniform(LN_DT_LO, LN_DT_HI, size=(batch, seqlen, nheads))).astype(np.float32)
    out["A"] = (-np.exp(rng.uniform(0.0, LN_A_HI, size=(nheads,)))).astype(np.float32)
    out["B"] = _normal(rng, (batch, seqlen, ngroups, dstate), dtype)
    out["C"] = _normal(rng, (batch, seqlen, ngroups, dstate), dtype)
    out["D"] = rng.standard_normal(size=(nheads,), dtype=np.float32) if with_D else None
    if random_init:
        out["init"] = (rng.standard_normal(size=(batch, nheads, headdim, dstate), dtype=np.float32)
                       * np.float32(0.1)).astype(np.float32)
    else:
        out["init"] = None
    return out


def scan_inputs_for(shape: ScanShape, seed=0):
    return scan_inputs(shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                       shape.dstate, shape.ngroups, shape.dtype, seed,
                       shape.random_init)


def packed_lengths(nseq, lo, hi, seed=0):
    """nseq sequence lengths, log-uniform in [lo, hi] (rounded down), a mix
    of short and long sequences for a packed batch."""
    rng = np.random.Generator(np.random.PCG64([seed, 7727]))
    return [int(v) for v in np.exp(rng.uniform(np.log(lo), np.log(hi + 1), size=nseq))
            .astype(np.int64).clip(lo, hi)]


def varlen_inputs(lengths, nheads, headdim, dstate, ngroups, dtype="bf16", seed=0,
                  random_init=False, with_D=True):
    """Inputs for a scan of packed sequences laid end to end, sequence s being
    tokens cu[s] .. cu[s+1]-1.  Token arrays are drawn as one scan_inputs row
    of T = sum(lengths) tokens.  Returns the scan_inputs keys with the batch
    axis dropped (x [T,H,P], dt [T,H], B, C [T,G,N]), init [nseq,H,P,N] (or
    None) and cu [nseq+1] int32."""
    lengths = [int(v) for v in lengths]
    T = sum(lengths)
    out = scan_inputs(1, T, nheads, headdim, dstate, ngroups, dtype, seed, False, with_D)
    for k in ("x", "dt", "B", "C"):
        out[k] = out[k][0]
    out["cu"] = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    if random_init:
        rng = np.random.Generator(np.random.PCG64([seed, 65537]))
        out["init"] = (rng.standard_normal(size=(len(lengths), nheads, headdim, dstate),
                                           dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    return out


def gate_input(shape, dtype="bf16", seed=0):
    """The output gate's z ~ N(0, 1) in the workload's input dtype (float32
    values, bf16-representable for bf16)."""
    rng = np.random.Generator(np.random.PCG64([seed, 31337]))
    return _normal(rng, tuple(shape), dtype)


def decode_params(nheads, seed=0):
    """Per-head A and D for a decode layer stack (float32)."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    A = (-np.exp(rng.uniform(0.0, LN_A_HI, size=(nheads,)))).astype(np.float32)
    D = rng.standard_normal(size=(nheads,), dtype=np.float32)
    return A, D


def decode_token_inputs(batch, nheads, headdim, dstate, ngroups, dtype="bf16",
                        seed=0, step=0):
    """Fresh per-token decode inputs: x [b,H,P], dt [b,H], B, C [b,G,N]."""
    rng = np.random.Generator(np.random.PCG64([seed, step, 104729]))
    out = {}
    out["x"] = _normal(rng, (batch, nheads, headdim), dtype)
    out["dt"] = np.exp(rng.uniform(LN_DT_LO, LN_DT_HI, size=(batch, nheads))).astype(np.float32)
    out["B"] = _normal(rng, (batch, ngroups, dstate), dtype)
    out["C"] = _normal(rng, (batch, ngroups, dstate), dtype)
    return out


def decode_state(batch, nheads, headdim, dstate, seed=0):
    """Host decode state ~ N(0, 1), float32 [b,H,P,N]."""
    rng = np.random.Generator(np.random.PCG64([seed, 15485863]))
    return rng.standard_normal(size=(batch, nheads, headdim, dstate), dtype=np.float32)


def device_decode_state(batch, nheads, headdim, dstate, seed=0, device="cuda"):
    """Decode state ~ N(0, 1) drawn on the device (for stacks too large to
    stage through the host).  Returns a float32 torch tensor [b,H,P,N]."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)
    return torch.randn((batch, nheads, headdim, dstate), generator=g,
                       device=device, dtype=torch.float32)


def device_decode_token_inputs(batch, nheads, headdim, dstate, ngroups, seed=0,
                               step=0, device="cuda"):
    """Per-token decode inputs drawn on the device (same distributions as
    ``decode_token_inputs``; bf16 x/B/C, float32 dt)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 7919 + int(step)) * 2 + 1)
    x = torch.randn((batch, nheads, headdim), generator=g, device=device).to(torch.bfloat16)
    u = torch.rand((batch, nheads), generator=g, device=device)
    dt = torch.exp(LN_DT_LO + (LN_DT_HI - LN_DT_LO) * u).to(torch.float32)
    B = torch.randn((batch, ngroups, dstate), generator=g, device=device).to(torch.bfloat16)
    C = torch.randn((batch, ngroups, dstate), generator=g, device=device).to(torch.bfloat16)
    return {"x": x, "dt": dt, "B": B, "C": C}
