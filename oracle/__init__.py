"""fp64 CPU oracle for the Mamba-2 SSD scan and decode step.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The library path never imports this
package, and this package imports nothing from the library.

The arithmetic lives in ``ssd_oracle.c`` (plain C, double precision, libm
``exp``); this module compiles it with gcc and marshals numpy arrays.  See the
header of ``ssd_oracle.c`` for the recurrence, the layouts and the pages each
step follows.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against the quadratic (dual) form, closed forms, a hand-derived example and
invariances; none is pinned by values printed on the pages, which print none.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c into libssd_oracle.so (gcc -O2, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_scan_seq.restype = ctypes.c_int
            lib.oracle_scan_seq.argtypes = [_dp] * 7 + [_i64] * 6 + [_dp, _dp, ctypes.c_int]
            lib.oracle_step.restype = ctypes.c_int
            lib.oracle_step.argtypes = [_dp] * 7 + [_i64] * 5 + [_dp, ctypes.c_int]
            lib.oracle_scan_chunked.restype = ctypes.c_int
            lib.oracle_scan_chunked.argtypes = ([_dp] * 7 + [_i64] * 7
                                                + [_dp] * 4 + [ctypes.c_int])
            _lib = lib
    return _lib


def _d(a):
    """C-contiguous float64 copy/view (exact for float32 and bf16 values)."""
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(_dp)


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def scan_seq(x, dt, A, B, C, D=None, init=None, nthreads=None):
    """Sequential recurrence.  x [b,L,H,P], dt [b,L,H], A [H], B/C [b,L,G,N],
    D [H] or None, init [b,H,P,N] or None.  Returns (y [b,L,H,P],
    final [b,H,P,N]) in float64."""
    x, dt, A, B, C = _d(x), _d(dt), _d(A), _d(B), _d(C)
    D = None if D is None else _d(D)
    init = None if init is None else _d(init)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.empty((b, L, H, P), np.float64)
    fin = np.empty((b, H, P, N), np.float64)
    rc = _load().oracle_scan_seq(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                 _ptr(D), _ptr(init), b, L, H, P, N, G,
                                 _ptr(y), _ptr(fin), _threads(nthreads))
    if rc:
        raise ValueError(f"oracle_scan_seq rejected its arguments (rc={rc})")
    return y, fin


def scan_varlen(x, dt, A, B, C, cu, D=None, init=None, nthreads=None):
    """Packed sequences: x [T,H,P], dt [T,H], B/C [T,G,N], cu [nseq+1]
    offsets (sequence s is tokens cu[s] .. cu[s+1]-1), init [nseq,H,P,N] or
    None.  Each sequence is the recurrence on its own from its own initial
    state (the pages define the scan per sequence; an empty one leaves its
    state as it was).  Returns (y [T,H,P], final [nseq,H,P,N]) in float64."""
    x, dt, B, C = _d(x), _d(dt), _d(B), _d(C)
    cu = [int(v) for v in np.asarray(cu)]
    nseq = len(cu) - 1
    T, H, P = x.shape
    N = B.shape[2]
    y = np.empty((T, H, P), np.float64)
    fin = np.zeros((nseq, H, P, N), np.float64)
    for s in range(nseq):
        a, b = cu[s], cu[s + 1]
        h0 = None if init is None else _d(init)[s:s + 1]
        if b == a:
            if h0 is not None:
                fin[s] = h0[0]
            continue
        ys, fs = scan_seq(x[None, a:b], dt[None, a:b], A, B[None, a:b], C[None, a:b],
                          D, h0, nthreads)
        y[a:b] = ys[0]
        fin[s] = fs[0]
    return y, fin


def step(state, x, dt, A, B, C, D=None, nthreads=None):
    """One decode token.  state [b,H,P,N] (not modified; a float64 copy is
    updated and returned), x [b,H,P], dt [b,H], B/C [b,G,N].  Returns
    (y [b,H,P], new_state [b,H,P,N])."""
    st = np.array(state, dtype=np.float64, order="C", copy=True)
    x, dt, A, B, C = _d(x), _d(dt), _d(A), _d(B), _d(C)
    D = None if D is None else _d(D)
    b, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    y = np.empty((b, H, P), np.float64)
    rc = _load().oracle_step(_ptr(st), _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                             _ptr(C), _ptr(D), b, H, P, N, G, _ptr(y),
                             _threads(nthreads))
    if rc:
        raise ValueError(f"oracle_step rejected its arguments (rc={rc})")
    return y, st


def scan_chunked(x, dt, A, B, C, chunk, D=None, init=None, nthreads=None,
                 want_intermediates=False):
    """The same scan computed chunk by chunk.  Returns (y, final) or, with
    want_intermediates, (y, final, S [b,nc,H,P,N], Hprev [b,nc,H,P,N]) where
    S is each chunk's own state contribution and Hprev the state entering it."""
    x, dt, A, B, C = _d(x), _d(dt), _d(A), _d(B), _d(C)
    D = None if D is None else _d(D)
    init = None if init is None else _d(init)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    nc = (L + chunk - 1) // chunk
    y = np.empty((b, L, H, P), np.float64)
    fin = np.empty((b, H, P, N), np.float64)
    S = Hp = None
    if want_intermediates:
        S = np.empty((b, nc, H, P, N), np.float64)
        Hp = np.empty((b, nc, H, P, N), np.float64)
    rc = _load().oracle_scan_chunked(_ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                     _ptr(C), _ptr(D), _ptr(init), b, L, H, P,
                                     N, G, chunk, _ptr(y), _ptr(fin), _ptr(S),
                                     _ptr(Hp), _threads(nthreads))
    if rc:
        raise ValueError(f"oracle_scan_chunked rejected its arguments (rc={rc})")
    if want_intermediates:
        return y, fin, S, Hp
    return y, fin


def dt_transform(dt, bias=None, softplus=False, lo=-np.inf, hi=np.inf):
    """The step size the kernels use when given a raw dt and a transform, in
    fp64: clamp(sp(dt + bias[h]), lo, hi) with sp(u) = log(1 + e^u) when
    ``softplus`` (evaluated as logaddexp(0, u), the same quantity without
    overflow), else sp(u) = u.  The head axis is dt's last axis.  The pages
    take the step from the input projection (CGLA section III.A) and do not
    say how it is made positive; this is the usual bias + softplus form."""
    u = np.asarray(dt, dtype=np.float64)
    if bias is not None:
        u = u + np.asarray(bias, dtype=np.float64)
    if softplus:
        u = np.logaddexp(0.0, u)
    return np.minimum(np.maximum(u, lo), hi)


def round_bf16(a):
    """Each value rounded to the nearest bfloat16 (8 significant bits), ties
    to even, returned as float64: the significand from frexp scaled to 8 bits
    and rounded half-to-even.  Finite normal values only."""
    m, e = np.frexp(np.asarray(a, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def decode_e4m3(codes):
    """8-bit E4M3 codes (uint8) -> their float64 values, from the format's
    definition: bit 7 the sign, bits 6..3 the exponent field e (bias 7), bits
    2..0 the significand field m.  e = 0 encodes the subnormals m * 2^-9
    (= (m / 8) * 2^(1 - 7)); e > 0 encodes (1 + m / 8) * 2^(e - 7), except
    that e = 15 with m = 7 is NaN (the encoding has no infinities, so the
    largest finite value is (1 + 6/8) * 2^8 = 448).  The pages name reduced
    precision as future work (CGLA sections V.A and VI) without a format;
    E4M3 is the common 8-bit floating-point one."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m, -9), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def step_bf16_state(state, x, dt, A, B, C, D=None, nthreads=None):
    """One decode token with the state stored in bfloat16: the fp64 step on
    the stored (bf16) state, y from the updated state before rounding, and
    the new state rounded to bf16.  The pages leave the reduced-precision
    format open (CGLA sections IV and VI); this is the plainest one."""
    y, st = step(state, x, dt, A, B, C, D, nthreads)
    return y, round_bf16(st)


def gate(y, z):
    """The output gate in fp64: y * silu(z), silu(z) = z * sigmoid(z), with
    sigmoid(z) = exp(-log(1 + e^-z)) (logaddexp, so no overflow).  The pages
    fuse the layer's neighbouring steps into the scan without spelling the
    gate out; this is the usual Mamba-2 form."""
    z = np.asarray(z, dtype=np.float64)
    return np.asarray(y, dtype=np.float64) * (z * np.exp(-np.logaddexp(0.0, -z)))


def rel_l2(got, ref):
    """||got - ref||_2 / ||ref||_2 in float64 (absolute norm when ref == 0)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = float(np.linalg.norm((got - ref).ravel()))
    den = float(np.linalg.norm(ref.ravel()))
    return num / den if den > 0 else num
