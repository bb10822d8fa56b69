"""Host-side pieces of bench.py (no GPU): the algorithmic work counts the
roofline divides by, the recorded DRAM traffic lookup, and the peak fallback."""
import json
import os

import bench
from state_space_model_chunked_gb300 import inputs as gen


def test_headline_algorithmic_bytes_and_flops():
    """130M layer, L 4096, H 24, P 64, N 128, G 1, Q 256, bf16, no init:
    bytes = x + y (2 each) + dt (4) + B + C (2 each) + A + D + final state;
    FLOPs = per chunk G Q(Q+1) N + H [Q(Q+1) P + 4 Q N P + 2 N P]."""
    s = gen.SCAN_SHAPES["mamba2_130m_L4096"]
    flops, byts = bench.scan_flops_bytes(s, s.random_init)
    L, H, P, N, Q = 4096, 24, 64, 128, 256
    want_b = 2 * L * H * P * 2 + L * H * 4 + 2 * L * N * 2 + 2 * H * 4 + H * P * N * 4
    assert byts == want_b == 28442816
    per_chunk = Q * (Q + 1) * N + H * (Q * (Q + 1) * P + 4 * Q * N * P + 2 * N * P)
    assert flops == (L // Q) * per_chunk


def test_recorded_traffic_is_tied_to_the_sources(tmp_path, monkeypatch):
    """The traffic figure is reported only while the kernel's sources hash as
    they did when it was captured."""
    import hashlib
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    rec = {"k": {"w": {"bytes_per_launch": 123, "sources": ["k.cu"],
                       "sources_sha256": hashlib.sha256(b"kernel v1").hexdigest()}}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("k", "w") == 123
    assert bench.ncu_traffic("k", "other") is None
    src.write_text("kernel v2")
    assert bench.ncu_traffic("k", "w") is None


def test_peaks_fall_back_when_unmeasured():
    peaks = bench.load_peaks()
    assert peaks["hbm_gbs"] > 0 and peaks["source"] in ("fallback", "measured")


def test_fp8_workload_bytes():
    """The long layer with E4M3 inputs: x, B, C one byte a value, y bf16 (two),
    dt, A, D and the final state as for bf16 inputs."""
    s8 = gen.SCAN_SHAPES["mamba2_2p7b_L65536_fp8"]
    s16 = gen.SCAN_SHAPES["mamba2_2p7b_L65536"]
    _, b8 = bench.scan_flops_bytes(s8, s8.random_init)
    _, b16 = bench.scan_flops_bytes(s16, s16.random_init)
    L, H, P, N = 65536, 80, 64, 128
    assert b16 - b8 == L * H * P + 2 * L * N       # one byte less per x, B, C value
    assert b8 == L * H * P * 3 + L * H * 4 + 2 * L * N + 2 * H * 4 + H * P * N * 4
