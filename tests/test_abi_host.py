"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/ssd.h declares, and rejects bad arguments
before enqueuing anything."""
import ctypes
import os
import re

import pytest

import state_space_model_chunked_gb300 as ssd
from state_space_model_chunked_gb300 import build as ssd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 5
FP8 = 2


@pytest.fixture(scope="module")
def lib():
    ssd_build.build()
    return ssd.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(ssd_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_binding_symbols():
    assert sorted(ssd.EXPORTED_SYMBOLS) == _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libssd.so does not export {name}"


def test_status_strings(lib):
    for code in range(6):
        s = lib.ssd_status_string(code).decode()
        assert s.startswith("SSD_")
    assert "UNKNOWN" in lib.ssd_status_string(99).decode()


def _fake(addr):
    return ctypes.c_void_p(addr)


def _scan(lib, **kw):
    a = dict(x=_fake(0x1000), dt=_fake(0x2000), A=_fake(0x3000), B=_fake(0x4000),
             C=_fake(0x5000), D=None, dtype=1, b=1, L=256, H=4, P=64, N=64, G=1, Q=64,
             init=None, y=_fake(0x6000), fin=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.ssd_scan_fwd(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["dtype"],
                            a["b"], a["L"], a["H"], a["P"], a["N"], a["G"], a["Q"],
                            a["init"], a["y"], a["fin"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(x=None), INVALID),
    (dict(dt=None), INVALID),
    (dict(y=None), INVALID),
    (dict(b=0), INVALID),
    (dict(L=-3), INVALID),
    (dict(H=6, G=4), INVALID),          # heads not a multiple of groups
    (dict(Q=48), INVALID),              # chunk not in {16,32,64,128,256}
    (dict(dtype=7), INVALID),
    (dict(x=_fake(0x1008)), INVALID),   # 8-byte aligned only
    (dict(fin=_fake(0x7004)), INVALID),
    (dict(N=66), UNSUPPORTED),          # dstate not a multiple of 4
    (dict(N=512), UNSUPPORTED),
])
def test_scan_rejects_bad_arguments(lib, kw, expect):
    assert _scan(lib, **kw) == expect


def test_scan_algo_rejects_unknown_algo(lib):
    a = [_fake(0x1000), _fake(0x2000), _fake(0x3000), _fake(0x4000), _fake(0x5000), None,
         1, 1, 256, 4, 64, 64, 1, 64, None, _fake(0x6000), None, None, 0, None]
    assert lib.ssd_scan_fwd_algo(9, *a) == INVALID


def _dec(lib, **kw):
    a = dict(state=_fake(0x1000), x=_fake(0x2000), dt=_fake(0x3000), A=_fake(0x4000),
             B=_fake(0x5000), C=_fake(0x6000), D=None, dtype=1, b=2, H=4, P=16, N=16, G=1,
             y=_fake(0x7000), stream=None)
    a.update(kw)
    return lib.ssd_state_update(a["state"], a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                                a["dtype"], a["b"], a["H"], a["P"], a["N"], a["G"], a["y"],
                                a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(state=None), INVALID),
    (dict(C=None), INVALID),
    (dict(H=0), INVALID),
    (dict(H=5, G=2), INVALID),
    (dict(B=_fake(0x5004)), INVALID),
    (dict(N=24), UNSUPPORTED),          # not a power of two
    (dict(N=512), UNSUPPORTED),
    (dict(N=2), UNSUPPORTED),
])
def test_decode_rejects_bad_arguments(lib, kw, expect):
    assert _dec(lib, **kw) == expect


def test_workspace_query_rejects_bad_sizes(lib):
    bad = ctypes.c_size_t(-1).value
    assert lib.ssd_scan_workspace_bytes(0, 256, 4, 64, 64, 1, 64) == bad
    assert lib.ssd_scan_workspace_bytes(1, 256, 6, 64, 64, 4, 64) == bad
    assert lib.ssd_scan_workspace_bytes(1, 256, 4, 64, 64, 1, 100) == bad
    assert lib.ssd_scan_fused_workspace_bytes(0, 256, 4, 64, 64, 1, 64, 1, 1) == bad
    assert lib.ssd_scan_fused_workspace_bytes(1, 256, 4, 64, 64, 1, 48, 1, 0) == bad
    # the fp32 path needs no workspace, with or without a dt transform
    assert lib.ssd_scan_fused_workspace_bytes(1, 256, 4, 64, 64, 1, 64, 0, 0) == 0
    assert lib.ssd_scan_fused_workspace_bytes(1, 256, 4, 64, 64, 1, 64, 0, 1) == 0


def test_fault_hook_rejects_unknown_fault(lib):
    assert lib.ssd_debug_inject_fault(7, 0) == INVALID
    assert lib.ssd_debug_inject_fault(0, 0) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 4, 2, 8)
    with pytest.raises((ValueError, ImportError)):
        ssd.scan_fwd(x, torch.zeros(1, 4, 2), torch.zeros(2), torch.zeros(1, 4, 1, 8),
                     torch.zeros(1, 4, 1, 8))


def _cu(vals):
    arr = (ctypes.c_int * len(vals))(*vals)
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def _varlen(lib, cu_vals, **kw):
    keep, cu = _cu(cu_vals)
    a = dict(algo=0, x=_fake(0x1000), dt=_fake(0x2000), A=_fake(0x3000), B=_fake(0x4000),
             C=_fake(0x5000), D=None, tr=None, z=None, dtype=1, nseq=len(cu_vals) - 1, cu=cu,
             cu_dev=_fake(0x8000), H=4, P=64, N=64, G=1, Q=64, init=None, y=_fake(0x6000),
             fin=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.ssd_scan_fwd_varlen(a["algo"], a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                                   a["tr"], a["z"], a["dtype"], a["nseq"], a["cu"], a["cu_dev"],
                                   a["H"], a["P"], a["N"], a["G"], a["Q"], a["init"], a["y"],
                                   a["fin"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("cu_vals,kw", [
    ([1, 5], {}),                        # offsets must start at 0
    ([0, 5, 3], {}),                     # and never decrease
    ([0, 5], dict(nseq=0)),
    ([0, 5], dict(cu=None)),
    ([0, 5], dict(cu_dev=None)),
    ([0, 5], dict(cu_dev=_fake(0x8002))),  # int-misaligned device offsets
    ([0, 5], dict(x=None)),              # tokens present: token arrays required
    ([0, 5], dict(H=6, G=4)),
    ([0, 5], dict(z=_fake(0x9008))),     # gate array 8-byte aligned only
])
def test_varlen_rejects_bad_arguments(lib, cu_vals, kw):
    assert _varlen(lib, cu_vals, **kw) == INVALID


def test_varlen_queries(lib):
    bad = ctypes.c_size_t(-1).value
    keep, cu = _cu([0, 3, 2])
    assert lib.ssd_scan_varlen_workspace_bytes(2, cu, 4, 64, 64, 1, 64, 1) == bad
    assert lib.ssd_scan_varlen_kernel_launches(2, cu, 4, 64, 64, 1, 64, 1) == -1
    keep, cu = _cu([0, 3, 9])
    assert lib.ssd_scan_varlen_workspace_bytes(2, cu, 4, 64, 64, 1, 64, 0) == 0   # fp32: SIMT
    assert lib.ssd_scan_varlen_kernel_launches(2, cu, 4, 64, 64, 1, 64, 0) == 1


def test_fused_scan_rejects_misaligned_gate(lib):
    a = [_fake(0x1000), _fake(0x2000), _fake(0x3000), _fake(0x4000), _fake(0x5000), None, None,
         _fake(0x9008), 1, 1, 256, 4, 64, 64, 1, 64, None, _fake(0x6000), None, None, 0, None]
    assert lib.ssd_scan_fwd_fused(0, *a) == INVALID


def _dec_fused(lib, **kw):
    a = dict(state=_fake(0x1000), sdt=0, x=_fake(0x2000), dt=_fake(0x3000), A=_fake(0x4000),
             B=_fake(0x5000), C=_fake(0x6000), D=None, tr=None, z=None, dtype=1, b=2, H=4, P=16,
             N=16, G=1, y=_fake(0x7000), stream=None)
    a.update(kw)
    return lib.ssd_state_update_fused(a["state"], a["sdt"], a["x"], a["dt"], a["A"], a["B"],
                                      a["C"], a["D"], a["tr"], a["z"], a["dtype"], a["b"],
                                      a["H"], a["P"], a["N"], a["G"], a["y"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(sdt=5), INVALID),                  # unknown state dtype
    (dict(sdt=1, dtype=0), UNSUPPORTED),     # bf16 state needs bf16 inputs
    (dict(z=_fake(0x9004)), INVALID),        # gate array not 16-byte aligned
    (dict(state=None), INVALID),
])
def test_fused_decode_rejects_bad_arguments(lib, kw, expect):
    assert _dec_fused(lib, **kw) == expect


def test_dt_transform_rejects_inverted_limits(lib):
    class Tr(ctypes.Structure):
        _fields_ = [("dt_bias", ctypes.c_void_p), ("softplus", ctypes.c_int),
                    ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float)]
    tr = Tr(None, 1, 0.5, 0.1)
    assert _dec_fused(lib, tr=ctypes.cast(ctypes.pointer(tr), ctypes.c_void_p)) == INVALID
    tr_nan = Tr(None, 1, float("nan"), 0.1)
    assert _dec_fused(lib, tr=ctypes.cast(ctypes.pointer(tr_nan), ctypes.c_void_p)) == INVALID


def test_binding_host_offsets_validation():
    import numpy as np
    import torch
    from state_space_model_chunked_gb300._binding import _host_offsets
    cu, ptr = _host_offsets([0, 3, 3, 10])
    assert cu.dtype == np.int32 and list(cu) == [0, 3, 3, 10] and ptr.value
    cu, _ = _host_offsets(torch.tensor([0, 5], dtype=torch.int64))
    assert list(cu) == [0, 5]
    for bad in ([0], [[0, 1]], [0, -1], [0, 2 ** 31]):
        with pytest.raises(ValueError):
            _host_offsets(bad)


def test_binding_refuses_cpu_tensors_for_packed_and_decode():
    import torch
    x = torch.zeros(4, 2, 8)
    with pytest.raises((ValueError, ImportError)):
        ssd.scan_fwd_varlen(x, torch.zeros(4, 2), torch.zeros(2), torch.zeros(4, 1, 8),
                            torch.zeros(4, 1, 8), [0, 4])
    with pytest.raises((ValueError, ImportError)):
        ssd.state_update(torch.zeros(1, 2, 8, 8), torch.zeros(1, 2, 8), torch.zeros(1, 2),
                         torch.zeros(2), torch.zeros(1, 1, 8), torch.zeros(1, 1, 8))


def test_plain_c_caller(tmp_path, lib):
    """A C program linked against libssd.so gets the same argument errors:
    the boundary needs neither Python nor torch."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = None
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            cuda_inc = os.path.join(cand, "include")
            break
    if cuda_inc is None:
        pytest.skip("CUDA headers not found")
    libdir = os.path.dirname(ssd.lib_path())
    exe = tmp_path / "c_abi_check"
    subprocess.run([cc, "-std=c11", "-O1", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", str(exe),
                    ssd.lib_path(), f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "c abi ok" in out.stdout


def _dec_multi(lib, **kw):
    a = dict(state=_fake(0x1000), sdt=0, x=_fake(0x2000), dt=_fake(0x3000), A=_fake(0x4000),
             B=_fake(0x5000), C=_fake(0x6000), D=None, tr=None, z=None, dtype=1, b=2, T=4, H=4,
             P=16, N=16, G=1, y=_fake(0x7000), stream=None)
    a.update(kw)
    return lib.ssd_state_update_multi(a["state"], a["sdt"], a["x"], a["dt"], a["A"], a["B"],
                                      a["C"], a["D"], a["tr"], a["z"], a["dtype"], a["b"],
                                      a["T"], a["H"], a["P"], a["N"], a["G"], a["y"],
                                      a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(T=0), INVALID),                    # no token
    (dict(x=None), INVALID),
    (dict(H=6, G=4), INVALID),
    (dict(sdt=1, dtype=0), UNSUPPORTED),     # bf16 state needs bf16 inputs
    (dict(N=24), UNSUPPORTED),               # dstate not a power of two
    (dict(P=65, N=128), UNSUPPORTED),        # more rows than the kernel keeps on chip
    (dict(P=129, N=64), UNSUPPORTED),
    (dict(P=257, N=32), UNSUPPORTED),
    (dict(P=513, N=16), UNSUPPORTED),
    (dict(P=513, N=8), UNSUPPORTED),
    (dict(P=513, N=4), UNSUPPORTED),
    (dict(P=65, N=256), UNSUPPORTED),
    (dict(z=_fake(0x8004)), INVALID),        # misaligned gate
])
def test_multi_token_decode_rejects_bad_arguments(lib, kw, expect):
    assert _dec_multi(lib, **kw) == expect


# ---------------------------------------------------------------- fp8 (E4M3) inputs
@pytest.mark.parametrize("kw,expect", [
    (dict(), WORKSPACE),                          # the bf16 copies need a workspace
    (dict(ws=_fake(0x9010), wsb=1 << 30), INVALID),   # workspace not 256-byte aligned
    (dict(x=_fake(0x1008)), INVALID),
    (dict(C=None), INVALID),
    (dict(N=66), UNSUPPORTED),
    (dict(H=6, G=4), INVALID),
])
def test_fp8_scan_checks_before_enqueueing(lib, kw, expect):
    assert _scan(lib, dtype=FP8, **kw) == expect


def test_fp8_workspace_adds_the_bf16_copies(lib):
    """fp8 calls need the bf16 call's workspace plus the bfloat16 copies of x,
    B and C (2 bytes a value, each rounded up to 256 bytes), and one launch
    more (the widening)."""
    def up(v):
        return (v + 255) // 256 * 256
    b, L, H, P, N, G = 2, 300, 4, 64, 64, 2
    copies = up(b * L * H * P * 2) + 2 * up(b * L * G * N * 2)
    for with_dt in (0, 1):
        assert (lib.ssd_scan_fused_workspace_bytes(b, L, H, P, N, G, 64, FP8, with_dt) ==
                copies + lib.ssd_scan_fused_workspace_bytes(b, L, H, P, N, G, 64, 1, with_dt))
    assert (lib.ssd_scan_kernel_launches(b, L, H, P, N, G, 64, FP8) ==
            1 + lib.ssd_scan_kernel_launches(b, L, H, P, N, G, 64, 1))
    keep, cu = _cu([0, 100, 100, 350])
    T = 350
    copies = up(T * H * P * 2) + 2 * up(T * G * N * 2)
    assert (lib.ssd_scan_varlen_workspace_bytes(3, cu, H, P, N, G, 64, FP8) ==
            copies + lib.ssd_scan_varlen_workspace_bytes(3, cu, H, P, N, G, 64, 1))
    assert (lib.ssd_scan_varlen_kernel_launches(3, cu, H, P, N, G, 64, FP8) ==
            1 + lib.ssd_scan_varlen_kernel_launches(3, cu, H, P, N, G, 64, 1))
    keep, cu = _cu([0, 0])              # no tokens: nothing to widen
    assert (lib.ssd_scan_varlen_workspace_bytes(1, cu, H, P, N, G, 64, FP8) ==
            lib.ssd_scan_varlen_workspace_bytes(1, cu, H, P, N, G, 64, 1))
    assert (lib.ssd_scan_varlen_kernel_launches(1, cu, H, P, N, G, 64, FP8) ==
            lib.ssd_scan_varlen_kernel_launches(1, cu, H, P, N, G, 64, 1))


def test_fp8_decode_is_unsupported(lib):
    assert _dec(lib, dtype=FP8) == UNSUPPORTED
    assert _dec_fused(lib, dtype=FP8) == UNSUPPORTED
    assert _dec_multi(lib, dtype=FP8) == UNSUPPORTED


def test_fp8_widening_checks(lib):
    w = lib.ssd_fp8_e4m3_to_bf16
    assert w(None, None, 0, None) == OK                       # nothing to do
    assert w(None, _fake(0x2000), 16, None) == INVALID
    assert w(_fake(0x1000), None, 16, None) == INVALID
    assert w(_fake(0x1001), _fake(0x2000), 16, None) == INVALID
    assert w(_fake(0x1000), _fake(0x2008), 16, None) == INVALID


def test_fp8_static_entry_rejects_copies_beyond_its_scratch(lib):
    """The built-in scratch (64 MiB) cannot hold the bfloat16 copies of the
    65536-token, 80-head layer's x (671 MB): SSD_ERR_WORKSPACE before any
    launch."""
    a = [_fake(0x1000), _fake(0x2000), _fake(0x3000), _fake(0x4000), _fake(0x5000), None,
         FP8, 1, 65536, 80, 64, 128, 1, 256, None, _fake(0x6000), None, None]
    assert lib.ssd_scan_fwd_static(*a) == WORKSPACE


def test_sequence_split_calls_reject_bad_arguments(lib):
    """The exchange of a sequence split over GPUs: null pointers, sizes <= 0
    and inverted transform limits come back before any launch."""
    dt, A, out = _fake(0x1000), _fake(0x2000), _fake(0x3000)
    assert lib.ssd_range_log_decay(None, A, None, 1, 16, 4, out, None) == INVALID
    assert lib.ssd_range_log_decay(dt, A, None, 1, 0, 4, out, None) == INVALID
    assert lib.ssd_range_log_decay(dt, A, None, 1, 16, 0, out, None) == INVALID
    assert lib.ssd_range_log_decay(dt, A, None, 1, 16, 4, None, None) == INVALID

    class Tr(ctypes.Structure):
        _fields_ = [("dt_bias", ctypes.c_void_p), ("softplus", ctypes.c_int),
                    ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float)]
    tr = Tr(None, 1, 0.5, 0.1)
    assert lib.ssd_range_log_decay(dt, A, ctypes.cast(ctypes.pointer(tr), ctypes.c_void_p),
                                   1, 16, 4, out, None) == INVALID
    c, d, e = _fake(0x4000), _fake(0x5000), _fake(0x6000)
    assert lib.ssd_chain_states(None, d, None, 2, 1, 4, 8, 8, e, None) == INVALID
    assert lib.ssd_chain_states(c, None, None, 2, 1, 4, 8, 8, e, None) == INVALID
    assert lib.ssd_chain_states(c, d, None, 2, 1, 4, 8, 8, None, None) == INVALID
    assert lib.ssd_chain_states(c, d, None, 0, 1, 4, 8, 8, e, None) == INVALID
    assert lib.ssd_chain_states(c, d, None, 2, 1, 4, 0, 8, e, None) == INVALID
