"""The scan entry point for callers that cannot allocate device memory
(ssd_scan_fwd_static): its scratch is an array built into the library, so a
caller whose memory is fixed up front -- an engine plugin handed only its
inputs and outputs, a runtime that forbids device allocation after start-up --
can still run long sequences.  Called through the C ABI and compared with
ssd_scan_fwd (caller-provided workspace) on two calls in a row with different
inputs, so the second call runs over the scratch the first one left behind.

This file is collected last so that a failure here cannot stop the rest of
the GPU suite early."""
import ctypes

import pytest
import torch

import state_space_model_chunked_gb300 as ssd
from state_space_model_chunked_gb300 import inputs as gen
from tests.gpu_util import TOL, dev, host, rel

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_static_scratch_scan_matches_workspace_scan_twice():
    lib = ssd.load()
    # 130M-shaped layer: long enough that the scan splits the sequence into
    # segments and needs scratch (checked below)
    b, L, H, P, N, G, Q = 1, 4096, 24, 64, 128, 1, 256
    need = ssd.scan_workspace_bytes(b, L, H, P, N, G, Q)
    assert 0 < need <= (32 << 20)
    stream = torch.cuda.current_stream()
    for seed in (101, 202):
        inp = gen.scan_inputs(b, L, H, P, N, G, "bf16", seed=seed, random_init=True)
        x, Bm, Cm = dev(inp["x"], "bf16"), dev(inp["B"], "bf16"), dev(inp["C"], "bf16")
        dt, A, D, init = dev(inp["dt"]), dev(inp["A"]), dev(inp["D"]), dev(inp["init"])
        y_ref, f_ref = ssd.scan_fwd(x, dt, A, Bm, Cm, D, Q, init)
        y = torch.empty_like(x)
        f = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
        rc = lib.ssd_scan_fwd_static(_ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                                     1, b, L, H, P, N, G, Q, _ptr(init), _ptr(y), _ptr(f),
                                     ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, lib.ssd_status_string(rc).decode()
        torch.cuda.synchronize()
        assert rel(host(y), host(y_ref)) <= TOL["bf16"]
        assert rel(host(f), host(f_ref)) <= TOL["bf16"]
    ssd.last_device_error()


def test_static_scratch_scan_rejects_shapes_beyond_its_scratch():
    lib = ssd.load()
    # the 2.7B-shaped 65536-token layer needs more scratch than the built-in array
    b, L, H, P, N, G, Q = 1, 65536, 80, 64, 128, 1, 256
    need = ssd.scan_workspace_bytes(b, L, H, P, N, G, Q)
    if need <= (32 << 20):
        pytest.skip("this device's segment plan fits the built-in scratch")
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: rejected before any launch
    rc = lib.ssd_scan_fwd_static(fake, fake, fake, fake, fake, None, 1, b, L, H, P, N, G, Q,
                                 None, fake, None, None)
    assert rc == 5   # SSD_ERR_WORKSPACE
