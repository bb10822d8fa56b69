"""GB300-native Mamba-2 state-space-duality (SSD) hot path.

A thin ctypes binding over ``libssd.so`` (C ABI in ``include/ssd.h``): it
checks tensor dtypes and devices, allocates outputs and workspace with torch,
passes raw device pointers and the current CUDA stream, and turns status codes
into exceptions.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback.  If the library is missing or
cannot load, every call raises.

    y, final = scan_fwd(x, dt, A, B, C, D, chunk=256, init_state=None)
    y, finals = scan_fwd_varlen(x, dt, A, B, C, cu_seqlens, D)   # packed sequences
    y, final = scan_fwd(x8, dt, A, B8, C8, D)           # float8_e4m3fn x/B/C -> bf16 y
    y = state_update(state, x, dt, A, B, C, D)          # state updated in place
    y = state_update_multi(state, x, dt, A, B, C, D)    # T tokens [b,T,H,P] in one call
    pipe = HostScanPipeline(); pipe.submit(..., out=(y_host, final_host))  # host tensors
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    HostScanPipeline,
    SsdError,
    lib_path,
    load,
    last_device_error,
    debug_inject_fault,
    FAULT_NONE,
    FAULT_WITHHOLD_SIGNAL,
    scan_fwd,
    scan_fwd_host,
    scan_fwd_varlen,
    scan_kernel_launches,
    scan_profile_events,
    scan_varlen_kernel_launches,
    scan_varlen_workspace_bytes,
    scan_workspace_bytes,
    state_update,
    state_update_multi,
    ALGO_AUTO,
    ALGO_SIMT,
    ALGO_TCGEN05,
    EXPORTED_SYMBOLS,
    FP8_E4M3,
    fp8_e4m3_to_bf16,
    range_log_decay,
    chain_states,
)
