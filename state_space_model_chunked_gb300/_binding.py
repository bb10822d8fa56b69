"""ctypes binding of libssd.so: argument marshalling only (see include/ssd.h)."""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libssd.so")

EXPORTED_SYMBOLS = (
    "ssd_scan_workspace_bytes",
    "ssd_scan_fused_workspace_bytes",
    "ssd_scan_kernel_launches",
    "ssd_scan_fwd",
    "ssd_scan_fwd_algo",
    "ssd_scan_fwd_dt",
    "ssd_scan_fwd_fused",
    "ssd_scan_fwd_static",
    "ssd_scan_fwd_varlen",
    "ssd_scan_varlen_workspace_bytes",
    "ssd_scan_varlen_kernel_launches",
    "ssd_scan_profile_events",
    "ssd_state_update",
    "ssd_state_update_dt",
    "ssd_state_update_fused",
    "ssd_state_update_multi",
    "ssd_status_string",
    "ssd_last_device_error",
    "ssd_debug_inject_fault",
    "ssd_fp8_e4m3_to_bf16",
    "ssd_range_log_decay",
    "ssd_chain_states",
)

ALGO_AUTO, ALGO_SIMT, ALGO_TCGEN05 = 0, 1, 2
_F32, _BF16, _FP8 = 0, 1, 2
# 8-bit E4M3 floats (prefill inputs x, B, C; see include/ssd.h)
FP8_E4M3 = torch.float8_e4m3fn

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_int = ctypes.c_int
_sz = ctypes.c_size_t


class _DtTransform(ctypes.Structure):
    """ssd_dt_transform: dt <- min(max(sp(dt + dt_bias[h]), dt_min), dt_max)."""
    _fields_ = [("dt_bias", ctypes.c_void_p), ("softplus", ctypes.c_int),
                ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float)]


class SsdError(RuntimeError):
    """A libssd.so call returned a non-OK status."""

    def __init__(self, fn, code, msg):
        super().__init__(f"{fn}: {msg} (status {code})")
        self.code = code


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libssd.so (built in-tree by state_space_model_chunked_gb300.build).
    Raises if it is missing: there is no fallback path."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"libssd.so not found at {_LIB_PATH}; build it with "
                "`python -m state_space_model_chunked_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.ssd_scan_workspace_bytes.restype = _sz
        lib.ssd_scan_workspace_bytes.argtypes = [_int] * 7
        lib.ssd_scan_fused_workspace_bytes.restype = _sz
        lib.ssd_scan_fused_workspace_bytes.argtypes = [_int] * 7 + [_int, _int]
        lib.ssd_debug_inject_fault.restype = _int
        lib.ssd_debug_inject_fault.argtypes = [_int, ctypes.c_ulonglong]
        lib.ssd_scan_kernel_launches.restype = _int
        lib.ssd_scan_kernel_launches.argtypes = [_int] * 7 + [_int]
        scan_args = [_vp] * 6 + [_int] * 8 + [_vp, _vp, _vp, _vp, _sz, _vp]
        lib.ssd_scan_fwd.restype = _int
        lib.ssd_scan_fwd.argtypes = scan_args
        lib.ssd_scan_fwd_algo.restype = _int
        lib.ssd_scan_fwd_algo.argtypes = [_int] + scan_args
        lib.ssd_scan_fwd_dt.restype = _int
        lib.ssd_scan_fwd_dt.argtypes = [_int] + [_vp] * 7 + [_int] * 8 + [_vp, _vp, _vp, _vp,
                                                                            _sz, _vp]
        lib.ssd_scan_fwd_fused.restype = _int
        lib.ssd_scan_fwd_fused.argtypes = [_int] + [_vp] * 8 + [_int] * 8 + [_vp, _vp, _vp, _vp,
                                                                               _sz, _vp]
        lib.ssd_scan_fwd_varlen.restype = _int
        lib.ssd_scan_fwd_varlen.argtypes = ([_int] + [_vp] * 8 + [_int, _int, _vp, _vp] +
                                            [_int] * 5 + [_vp, _vp, _vp, _vp, _sz, _vp])
        lib.ssd_scan_varlen_workspace_bytes.restype = _sz
        lib.ssd_scan_varlen_workspace_bytes.argtypes = [_int, _vp] + [_int] * 6
        lib.ssd_scan_varlen_kernel_launches.restype = _int
        lib.ssd_scan_varlen_kernel_launches.argtypes = [_int, _vp] + [_int] * 6
        lib.ssd_state_update_dt.restype = _int
        lib.ssd_state_update_dt.argtypes = [_vp] * 8 + [_int] * 6 + [_vp, _vp]
        lib.ssd_state_update_fused.restype = _int
        lib.ssd_state_update_fused.argtypes = [_vp, _int] + [_vp] * 8 + [_int] * 6 + [_vp, _vp]
        lib.ssd_state_update_multi.restype = _int
        lib.ssd_state_update_multi.argtypes = [_vp, _int] + [_vp] * 8 + [_int] * 7 + [_vp, _vp]
        lib.ssd_scan_fwd_static.restype = _int
        lib.ssd_scan_fwd_static.argtypes = [_vp] * 6 + [_int] * 8 + [_vp, _vp, _vp, _vp]
        lib.ssd_scan_profile_events.restype = _int
        lib.ssd_scan_profile_events.argtypes = [_vp, _vp]
        lib.ssd_state_update.restype = _int
        lib.ssd_state_update.argtypes = [_vp] * 7 + [_int] * 6 + [_vp, _vp]
        lib.ssd_status_string.restype = ctypes.c_char_p
        lib.ssd_status_string.argtypes = [_int]
        lib.ssd_last_device_error.restype = _int
        lib.ssd_last_device_error.argtypes = []
        lib.ssd_fp8_e4m3_to_bf16.restype = _int
        lib.ssd_fp8_e4m3_to_bf16.argtypes = [_vp, _vp, _sz, _vp]
        lib.ssd_range_log_decay.restype = _int
        lib.ssd_range_log_decay.argtypes = [_vp, _vp, _vp, _int, _int, _int, _vp, _vp]
        lib.ssd_chain_states.restype = _int
        lib.ssd_chain_states.argtypes = [_vp, _vp, _vp] + [_int] * 5 + [_vp, _vp]
        _lib = lib
        return lib


def _check(fn, code):
    if code != 0:
        msg = load().ssd_status_string(code).decode()
        raise SsdError(fn, code, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t):
    if t.dtype == torch.float32:
        return _F32
    if t.dtype == torch.bfloat16:
        return _BF16
    if t.dtype == FP8_E4M3:
        return _FP8
    raise TypeError(f"x/B/C must be float32, bfloat16 or float8_e4m3fn, got {t.dtype}")


def _code_of(dtype):
    """ssd_dtype code of a torch dtype given to the size queries."""
    return {torch.bfloat16: _BF16, FP8_E4M3: _FP8}.get(dtype, _F32)


def _out_dtype(x):
    """dtype of y (and of the gate's z) for inputs of x's dtype: bfloat16 for
    fp8 inputs, x's own otherwise."""
    return torch.bfloat16 if x.dtype == FP8_E4M3 else x.dtype


def _need(t, name, dtype=None, device=None, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def scan_workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups, chunk,
                         dtype=torch.bfloat16, device=None, dt_transform=False):
    """Workspace bytes of a scan_fwd call of this shape and input dtype on
    the device, with or without a dt transform."""
    lib = load()
    code = _code_of(dtype)
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        n = lib.ssd_scan_fused_workspace_bytes(batch, seqlen, nheads, headdim, dstate,
                                               ngroups, chunk, code, 1 if dt_transform else 0)
    if n == ctypes.c_size_t(-1).value:
        raise SsdError("ssd_scan_fused_workspace_bytes", 1, "invalid sizes")
    return int(n)


def scan_kernel_launches(batch, seqlen, nheads, headdim, dstate, ngroups, chunk,
                         dtype=torch.bfloat16, device=None):
    """Kernels one scan_fwd call enqueues for this shape on the device."""
    lib = load()
    code = _code_of(dtype)
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        n = lib.ssd_scan_kernel_launches(batch, seqlen, nheads, headdim, dstate, ngroups,
                                         chunk, code)
    if n < 0:
        raise SsdError("ssd_scan_kernel_launches", 1, "invalid sizes")
    return int(n)


def scan_varlen_workspace_bytes(cu_seqlens, nheads, headdim, dstate, ngroups, chunk,
                                dtype=torch.bfloat16, device=None):
    """Workspace bytes of scan_fwd_varlen for these offsets on the device."""
    lib = load()
    cu, cu_ptr = _host_offsets(cu_seqlens)
    code = _code_of(dtype)
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        n = lib.ssd_scan_varlen_workspace_bytes(cu.size - 1, cu_ptr, nheads, headdim, dstate,
                                                ngroups, chunk, code)
    if n == ctypes.c_size_t(-1).value:
        raise SsdError("ssd_scan_varlen_workspace_bytes", 1, "invalid sizes or offsets")
    return int(n)


def scan_varlen_kernel_launches(cu_seqlens, nheads, headdim, dstate, ngroups, chunk,
                                dtype=torch.bfloat16, device=None):
    """Kernels one scan_fwd_varlen call enqueues for these offsets."""
    lib = load()
    cu, cu_ptr = _host_offsets(cu_seqlens)
    code = _code_of(dtype)
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        n = lib.ssd_scan_varlen_kernel_launches(cu.size - 1, cu_ptr, nheads, headdim, dstate,
                                                ngroups, chunk, code)
    if n < 0:
        raise SsdError("ssd_scan_varlen_kernel_launches", 1, "invalid sizes or offsets")
    return int(n)


def _dt_transform(dt_bias, dt_softplus, dt_limit, H, dev):
    """A ctypes ssd_dt_transform for the keyword arguments, or None (identity)
    when none is set; the second value keeps dt_bias alive for the call."""
    if dt_bias is None and not dt_softplus and dt_limit is None:
        return None, None
    if dt_bias is not None:
        _need(dt_bias, "dt_bias", torch.float32, dev, (H,))
    lo, hi = dt_limit if dt_limit is not None else (float("-inf"), float("inf"))
    t = _DtTransform(dt_bias.data_ptr() if dt_bias is not None else None,
                     1 if dt_softplus else 0, lo, hi)
    return ctypes.byref(t), (t, dt_bias)


def scan_fwd(x, dt, A, B, C, D=None, chunk=256, init_state=None, *, y=None,
             final_state=None, workspace=None, algo=ALGO_AUTO, return_final=True,
             dt_bias=None, dt_softplus=False, dt_limit=None, z=None):
    """Chunked SSD scan (prefill).  x [b,L,H,P], dt [b,L,H] f32, A [H] f32,
    B/C [b,L,G,N] (x's dtype: float32, bfloat16 or float8_e4m3fn), D [H] f32 or
    None, init_state [b,H,P,N] f32 or None.  fp8 inputs give a bfloat16 y
    (the call widens them exactly to bfloat16 in its workspace).  dt_bias [H] f32, dt_softplus and dt_limit = (lo, hi) transform the
    raw dt inside the kernels: dt <- clamp(softplus(dt + dt_bias), lo, hi)
    (softplus only when dt_softplus).  z (x's shape and dtype) gates the
    output inside the kernels: y <- y * silu(z).  Returns (y, final_state) on
    x's device and the current stream."""
    lib = load()
    _need(x, "x")
    dev = x.device
    b, L, H, P = x.shape
    _need(B, "B", x.dtype, dev)
    G, N = B.shape[2], B.shape[3]
    _need(dt, "dt", torch.float32, dev, (b, L, H))
    _need(A, "A", torch.float32, dev, (H,))
    _need(B, "B", x.dtype, dev, (b, L, G, N))
    _need(C, "C", x.dtype, dev, (b, L, G, N))
    if D is not None:
        _need(D, "D", torch.float32, dev, (H,))
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, dev, (b, H, P, N))
    if z is not None:
        _need(z, "z", _out_dtype(x), dev, x.shape)
    if y is None:
        y = torch.empty(x.shape, dtype=_out_dtype(x), device=dev)
    else:
        _need(y, "y", _out_dtype(x), dev, x.shape)
    if final_state is None and return_final:
        final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=dev)
    elif final_state is not None:
        _need(final_state, "final_state", torch.float32, dev, (b, H, P, N))
    code = _dtype_code(x)
    with_dt = dt_bias is not None or dt_softplus or dt_limit is not None
    with torch.cuda.device(dev):
        need = lib.ssd_scan_fused_workspace_bytes(b, L, H, P, N, G, chunk, code,
                                                  1 if with_dt else 0)
        if need == ctypes.c_size_t(-1).value:
            raise SsdError("ssd_scan_fused_workspace_bytes", 1, "invalid sizes")
        if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        stream = torch.cuda.current_stream(dev).cuda_stream
        tptr, _keep = _dt_transform(dt_bias, dt_softplus, dt_limit, H, dev)
        rc = lib.ssd_scan_fwd_fused(algo, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                    _ptr(D), tptr, _ptr(z), code, b, L, H, P, N, G, chunk,
                                    _ptr(init_state), _ptr(y), _ptr(final_state),
                                    _ptr(workspace), wbytes, ctypes.c_void_p(stream))
    _check("ssd_scan_fwd", rc)
    return y, final_state


def _host_offsets(cu_seqlens):
    """(numpy int32 host copy, ctypes pointer) of packed sequence offsets."""
    import numpy as np
    if isinstance(cu_seqlens, torch.Tensor):
        cu_seqlens = cu_seqlens.detach().cpu().numpy()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    if cu.ndim != 1 or cu.size < 2:
        raise ValueError("cu_seqlens must hold nseq + 1 offsets")
    if cu.max() >= 2 ** 31 or cu.min() < 0:
        raise ValueError("cu_seqlens out of the int32 range")
    cu = cu.astype(np.int32)
    return cu, cu.ctypes.data_as(ctypes.c_void_p)


def scan_fwd_varlen(x, dt, A, B, C, cu_seqlens, D=None, chunk=256, init_state=None, *,
                    y=None, final_state=None, workspace=None, algo=ALGO_AUTO,
                    return_final=True, dt_bias=None, dt_softplus=False, dt_limit=None,
                    z=None, cu_seqlens_dev=None):
    """Scan of nseq packed sequences.  x [T,H,P], dt [T,H] f32, B/C [T,G,N];
    cu_seqlens: nseq + 1 token offsets (a list, numpy array or tensor; 0 first,
    non-decreasing; sequence s is tokens cu[s]..cu[s+1]-1).  init_state and the
    returned final_state are [nseq,H,P,N] f32.  ``cu_seqlens_dev`` (int32 on
    x's device, same values) saves the host-to-device copy of the offsets.
    dt transform and gate (z [T,H,P]) keywords as scan_fwd.  Returns (y, final_state)."""
    lib = load()
    _need(x, "x")
    dev = x.device
    T, H, P = x.shape
    _need(B, "B", x.dtype, dev)
    G, N = B.shape[1], B.shape[2]
    cu, cu_ptr = _host_offsets(cu_seqlens)
    nseq = cu.size - 1
    if int(cu[-1]) != T:
        raise ValueError(f"cu_seqlens ends at {int(cu[-1])}, x holds {T} tokens")
    _need(dt, "dt", torch.float32, dev, (T, H))
    _need(A, "A", torch.float32, dev, (H,))
    _need(B, "B", x.dtype, dev, (T, G, N))
    _need(C, "C", x.dtype, dev, (T, G, N))
    if D is not None:
        _need(D, "D", torch.float32, dev, (H,))
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, dev, (nseq, H, P, N))
    if z is not None:
        _need(z, "z", _out_dtype(x), dev, x.shape)
    if y is None:
        y = torch.empty(x.shape, dtype=_out_dtype(x), device=dev)
    else:
        _need(y, "y", _out_dtype(x), dev, x.shape)
    if final_state is None and return_final:
        final_state = torch.empty((nseq, H, P, N), dtype=torch.float32, device=dev)
    elif final_state is not None:
        _need(final_state, "final_state", torch.float32, dev, (nseq, H, P, N))
    if cu_seqlens_dev is None:
        cu_seqlens_dev = torch.from_numpy(cu).to(dev, non_blocking=False)
    else:
        _need(cu_seqlens_dev, "cu_seqlens_dev", torch.int32, dev, (nseq + 1,))
    code = _dtype_code(x)
    with torch.cuda.device(dev):
        need = lib.ssd_scan_varlen_workspace_bytes(nseq, cu_ptr, H, P, N, G, chunk, code)
        if need == ctypes.c_size_t(-1).value:
            raise SsdError("ssd_scan_varlen_workspace_bytes", 1, "invalid sizes or offsets")
        if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        stream = torch.cuda.current_stream(dev).cuda_stream
        tptr, _keep = _dt_transform(dt_bias, dt_softplus, dt_limit, H, dev)
        rc = lib.ssd_scan_fwd_varlen(algo, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                     _ptr(D), tptr, _ptr(z), code, nseq, cu_ptr,
                                     _ptr(cu_seqlens_dev),
                                     H, P, N, G, chunk, _ptr(init_state), _ptr(y),
                                     _ptr(final_state), _ptr(workspace), wbytes,
                                     ctypes.c_void_p(stream))
    _check("ssd_scan_fwd_varlen", rc)
    return y, final_state


def scan_fwd_host(x, dt, A, B, C, D=None, chunk=256, init_state=None, *, device="cuda",
                  staging=None, out=None):
    """Scan with HOST (CPU) tensors: copies the inputs to the device, runs
    ssd_scan_fwd there and copies y and the final state back.  ``staging`` (a
    dict) keeps device buffers between calls; ``out`` = (y_host, final_host)
    receives the results (pinned for asynchronous copies).  Returns the host
    (y, final_state) after the stream has finished."""
    dev = torch.device(device)
    st = staging if staging is not None else {}
    host = {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D, "init": init_state}
    devt = {}
    for k, v in host.items():
        if v is None:
            devt[k] = None
            continue
        buf = st.get(k)
        if buf is None or buf.shape != v.shape or buf.dtype != v.dtype:
            buf = torch.empty(v.shape, dtype=v.dtype, device=dev)
            st[k] = buf
        buf.copy_(v, non_blocking=True)
        devt[k] = buf
    yd, fd = scan_fwd(devt["x"], devt["dt"], devt["A"], devt["B"], devt["C"], devt["D"],
                      chunk, devt["init"], y=st.get("y"), final_state=st.get("final"),
                      workspace=st.get("ws"))
    st["y"], st["final"] = yd, fd
    if out is None:
        out = (torch.empty(yd.shape, dtype=yd.dtype, pin_memory=True),
               torch.empty(fd.shape, dtype=fd.dtype, pin_memory=True))
    out[0].copy_(yd, non_blocking=True)
    out[1].copy_(fd, non_blocking=True)
    torch.cuda.current_stream(dev).synchronize()
    return out


class HostScanPipeline:
    """ssd_scan_fwd on host (CPU) tensors with the copies of consecutive calls
    overlapped: the inputs of call k+1 go to the device on one stream while
    call k computes on a second and the outputs of call k-1 come back on a
    third (the two copy directions use the link's two directions).  ``depth``
    staging slots of device buffers rotate; events order every reuse of a
    slot.  ``submit`` enqueues one call and returns at once; ``synchronize``
    waits for every call submitted so far.  Host tensors should be pinned."""

    def __init__(self, device="cuda", depth=2):
        self.dev = torch.device(device)
        self.depth = depth
        self.s_in = torch.cuda.Stream(self.dev)
        self.s_comp = torch.cuda.Stream(self.dev)
        self.s_out = torch.cuda.Stream(self.dev)
        self.slots = [{"loaded": torch.cuda.Event(), "computed": torch.cuda.Event(),
                       "drained": torch.cuda.Event()} for _ in range(depth)]
        self.ws = None
        self.n = 0

    def submit(self, x, dt, A, B, C, D=None, chunk=256, init_state=None, *, out):
        """Enqueue one call; ``out`` = (y_host, final_host) receives its results
        once ``synchronize`` (or the returned event) has completed."""
        st = self.slots[self.n % self.depth]
        host = {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D, "init": init_state}
        devt = {}
        # inputs: the slot's buffers are free once its previous call has computed
        self.s_in.wait_event(st["computed"])
        with torch.cuda.stream(self.s_in):
            for k, v in host.items():
                if v is None:
                    devt[k] = None
                    continue
                buf = st.get(k)
                if buf is None or buf.shape != v.shape or buf.dtype != v.dtype:
                    buf = torch.empty(v.shape, dtype=v.dtype, device=self.dev)
                    st[k] = buf
                buf.copy_(v, non_blocking=True)
                devt[k] = buf
            st["loaded"].record(self.s_in)
        # compute: inputs landed, and the slot's previous outputs have been read back
        self.s_comp.wait_event(st["loaded"])
        self.s_comp.wait_event(st["drained"])
        with torch.cuda.stream(self.s_comp):
            if self.ws is None:
                b, L, H, P = x.shape
                nbytes = scan_workspace_bytes(b, L, H, P, B.shape[3], B.shape[2], chunk,
                                              dtype=x.dtype, device=self.dev)
                self.ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=self.dev)
            yd, fd = scan_fwd(devt["x"], devt["dt"], devt["A"], devt["B"], devt["C"], devt["D"],
                              chunk, devt["init"], y=st.get("y"), final_state=st.get("final"),
                              workspace=self.ws)
            st["y"], st["final"] = yd, fd
            st["computed"].record(self.s_comp)
        # outputs back to the host
        self.s_out.wait_event(st["computed"])
        with torch.cuda.stream(self.s_out):
            out[0].copy_(yd, non_blocking=True)
            out[1].copy_(fd, non_blocking=True)
            st["drained"].record(self.s_out)
        self.n += 1
        return st["drained"]

    def synchronize(self):
        for s in (self.s_in, self.s_comp, self.s_out):
            s.synchronize()


def state_update(state, x, dt, A, B, C, D=None, *, y=None, dt_bias=None, dt_softplus=False,
                 dt_limit=None, z=None):
    """One decode token.  state [b,H,P,N] f32 or bf16 (updated in place; a
    bf16 state needs bf16 inputs and is rounded to nearest even after each
    fp32 update), x [b,H,P], dt [b,H] f32, A [H] f32, B/C [b,G,N] (x's dtype),
    D [H] f32 or None; dt_bias / dt_softplus / dt_limit and the gate
    z [b,H,P] as in scan_fwd.  Returns y [b,H,P] in x's dtype."""
    lib = load()
    _need(state, "state")
    if state.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"state must be float32 or bfloat16, got {state.dtype}")
    dev = state.device
    b, H, P, N = state.shape
    _need(x, "x", None, dev, (b, H, P))
    _need(dt, "dt", torch.float32, dev, (b, H))
    _need(A, "A", torch.float32, dev, (H,))
    _need(B, "B", x.dtype, dev)
    G = B.shape[1]
    _need(B, "B", x.dtype, dev, (b, G, N))
    _need(C, "C", x.dtype, dev, (b, G, N))
    if D is not None:
        _need(D, "D", torch.float32, dev, (H,))
    if z is not None:
        _need(z, "z", x.dtype, dev, (b, H, P))
    if y is None:
        y = torch.empty_like(x)
    else:
        _need(y, "y", x.dtype, dev, (b, H, P))
    code = _dtype_code(x)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        tptr, _keep = _dt_transform(dt_bias, dt_softplus, dt_limit, H, dev)
        rc = lib.ssd_state_update_fused(_ptr(state), _dtype_code(state), _ptr(x), _ptr(dt),
                                        _ptr(A), _ptr(B), _ptr(C), _ptr(D), tptr, _ptr(z), code,
                                        b, H, P, N, G, _ptr(y), ctypes.c_void_p(stream))
    _check("ssd_state_update", rc)
    return y


def state_update_multi(state, x, dt, A, B, C, D=None, *, y=None, dt_bias=None,
                       dt_softplus=False, dt_limit=None, z=None):
    """`ntokens` decode tokens per (batch, head) in one call (the state is
    read and written once).  state [b,H,P,N] f32 or bf16 (in place; a bf16
    state is rounded once, after the last token), x [b,T,H,P], dt [b,T,H]
    f32, A [H] f32, B/C [b,T,G,N] (x's dtype), D [H] f32 or None; the dt
    transform and gate z [b,T,H,P] as in state_update.  Returns y [b,T,H,P]."""
    lib = load()
    _need(state, "state")
    if state.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"state must be float32 or bfloat16, got {state.dtype}")
    dev = state.device
    b, H, P, N = state.shape
    _need(x, "x", None, dev)
    if x.dim() != 4 or x.shape[0] != b or x.shape[2] != H or x.shape[3] != P:
        raise ValueError(f"x has shape {tuple(x.shape)}, expected ({b}, T, {H}, {P})")
    T = x.shape[1]
    _need(dt, "dt", torch.float32, dev, (b, T, H))
    _need(A, "A", torch.float32, dev, (H,))
    _need(B, "B", x.dtype, dev)
    G = B.shape[2]
    _need(B, "B", x.dtype, dev, (b, T, G, N))
    _need(C, "C", x.dtype, dev, (b, T, G, N))
    if D is not None:
        _need(D, "D", torch.float32, dev, (H,))
    if z is not None:
        _need(z, "z", x.dtype, dev, x.shape)
    if y is None:
        y = torch.empty_like(x)
    else:
        _need(y, "y", x.dtype, dev, x.shape)
    code = _dtype_code(x)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        tptr, _keep = _dt_transform(dt_bias, dt_softplus, dt_limit, H, dev)
        rc = lib.ssd_state_update_multi(_ptr(state), _dtype_code(state), _ptr(x), _ptr(dt),
                                        _ptr(A), _ptr(B), _ptr(C), _ptr(D), tptr, _ptr(z), code,
                                        b, T, H, P, N, G, _ptr(y), ctypes.c_void_p(stream))
    _check("ssd_state_update_multi", rc)
    return y


def fp8_e4m3_to_bf16(src, out=None):
    """Widens a float8_e4m3fn (or uint8 holding E4M3 codes) CUDA tensor to
    bfloat16, exactly, in the library's kernel; returns the bfloat16 tensor."""
    lib = load()
    _need(src, "src")
    if src.dtype not in (FP8_E4M3, torch.uint8):
        raise TypeError(f"src must be float8_e4m3fn or uint8, got {src.dtype}")
    if out is None:
        out = torch.empty(src.shape, dtype=torch.bfloat16, device=src.device)
    else:
        _need(out, "out", torch.bfloat16, src.device, src.shape)
    with torch.cuda.device(src.device):
        stream = torch.cuda.current_stream(src.device).cuda_stream
        rc = lib.ssd_fp8_e4m3_to_bf16(_ptr(src), _ptr(out), src.numel(), ctypes.c_void_p(stream))
    _check("ssd_fp8_e4m3_to_bf16", rc)
    return out


def range_log_decay(dt, A, *, dt_bias=None, dt_softplus=False, dt_limit=None):
    """A token range's log-decay, [b, H] f32: A[h] times the sum of dt over
    the range (dt [b, L, H] f32, transformed as scan_fwd would with the same
    keywords).  One factor of the exchange when a sequence is split over GPUs."""
    lib = load()
    _need(dt, "dt", torch.float32)
    dev = dt.device
    b, L, H = dt.shape
    _need(A, "A", torch.float32, dev, (H,))
    out = torch.empty((b, H), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        tptr, _keep = _dt_transform(dt_bias, dt_softplus, dt_limit, H, dev)
        rc = lib.ssd_range_log_decay(_ptr(dt), _ptr(A), tptr, b, L, H, _ptr(out),
                                     ctypes.c_void_p(stream))
    _check("ssd_range_log_decay", rc)
    return out


def chain_states(contrib, log_decay, init=None):
    """Entering states [R, b, H, P, N] f32 of R consecutive token ranges:
    entering[0] = init (zeros when None), entering[r+1] = exp(log_decay[r])
    entering[r] + contrib[r], from contrib [R, b, H, P, N] (each range's state
    from a zero start) and log_decay [R, b, H]."""
    lib = load()
    _need(contrib, "contrib", torch.float32)
    dev = contrib.device
    R, b, H, P, N = contrib.shape
    _need(log_decay, "log_decay", torch.float32, dev, (R, b, H))
    if init is not None:
        _need(init, "init", torch.float32, dev, (b, H, P, N))
    out = torch.empty_like(contrib)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        rc = lib.ssd_chain_states(_ptr(contrib), _ptr(log_decay), _ptr(init), R, b, H, P, N,
                                  _ptr(out), ctypes.c_void_p(stream))
    _check("ssd_chain_states", rc)
    return out


def scan_profile_events(before=None, after=None):
    """Record torch.cuda.Event `before`/`after` around the y-writing kernel of
    every following scan_fwd call (None, None to stop).  The events must have
    been created on the device (record them once first)."""
    lib = load()
    if before is None or after is None:
        lib.ssd_scan_profile_events(None, None)
    else:
        lib.ssd_scan_profile_events(ctypes.c_void_p(before.cuda_event),
                                    ctypes.c_void_p(after.cuda_event))


def last_device_error():
    """Reads and clears the device error word (synchronises the device)."""
    rc = load().ssd_last_device_error()
    _check("ssd_last_device_error", rc)


FAULT_NONE, FAULT_WITHHOLD_SIGNAL = 0, 1


def debug_inject_fault(fault=FAULT_NONE, wait_limit_ns=0):
    """Test hook of the bounded device waits (ssd_debug_inject_fault):
    FAULT_WITHHOLD_SIGNAL makes the next tensor-core scans time out after
    wait_limit_ns; FAULT_NONE (and 0 = the default limit) restores them."""
    _check("ssd_debug_inject_fault", load().ssd_debug_inject_fault(int(fault), int(wait_limit_ns)))
