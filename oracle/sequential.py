"""ctypes front-end of the sequential float64 oracle (``ssd_oracle.c``).

TEST INFRASTRUCTURE ONLY.

The C code is the literal loop over time (Mamba-3-Lite "SSD Reference",
section "ssd_naive_complex -- the O(T) oracle": the oracle is a plain walk over
the sequence carrying one state per head) applied to the real Mamba-2
recurrence with the dt factor on the input, the D skip, the silu(z) gate and
initial/final states.  The backward is the exact adjoint of that loop.

Pinned by tests/test_oracle_pins.py (quadratic form, closed-form geometric
series, chunk-size and split invariance, linearity, scipy lfilter) and
tests/test_oracle_grad.py (central finite differences, torch float64 autograd of
the independent quadratic form).

All arrays are float64, token-major on a flat token axis:
  x, z, y, dx, dz : [T, H, P]      dt_raw, ddt_raw : [T, H]
  B, C, dB, dC    : [T, G, N]      A, D, dt_bias   : [H]
  init, final     : [S, H, P, N]   cu              : [S+1] int64 token offsets
"""
import ctypes
import os

import numpy as np

from . import build as _build, LIB_PATH

_lib = None


class _In(ctypes.Structure):
    _fields_ = [
        ("nseq", ctypes.c_int64), ("H", ctypes.c_int64), ("P", ctypes.c_int64),
        ("G", ctypes.c_int64), ("N", ctypes.c_int64),
        ("cu", ctypes.c_void_p), ("x", ctypes.c_void_p), ("dt_raw", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("Bm", ctypes.c_void_p), ("Cm", ctypes.c_void_p),
        ("D", ctypes.c_void_p), ("z", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("init", ctypes.c_void_p), ("head_mask", ctypes.c_void_p),
    ]


def _load():
    global _lib
    if _lib is None:
        _build()
        lib = ctypes.CDLL(LIB_PATH)
        lib.ssd_oracle_fwd.restype = ctypes.c_int
        lib.ssd_oracle_fwd.argtypes = [ctypes.POINTER(_In), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.ssd_oracle_bwd.restype = ctypes.c_int
        lib.ssd_oracle_bwd.argtypes = [ctypes.POINTER(_In)] + [ctypes.c_void_p] * 11 + [ctypes.c_int64, ctypes.c_int]
        lib.ssd_oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().ssd_oracle_num_threads())


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _make_in(x, dt_raw, A, B, C, D, z, dt_bias, init, cu, heads):
    x = _f64(x)
    T, H, P = x.shape
    B = _f64(B)
    G, N = B.shape[1], B.shape[2]
    if cu is None:
        cu = np.array([0, T], dtype=np.int64)
    cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int64))
    S = cu.shape[0] - 1
    mask = None
    if heads is not None:
        mask = np.zeros(H, dtype=np.int32)
        mask[np.asarray(heads)] = 1
    arrs = dict(x=x, dt_raw=_f64(dt_raw), A=_f64(A), B=B, C=_f64(C), D=_f64(D), z=_f64(z),
                dt_bias=_f64(dt_bias), init=_f64(init), cu=cu, mask=mask)
    s = _In(S, H, P, G, N, _ptr(cu), _ptr(arrs["x"]), _ptr(arrs["dt_raw"]), _ptr(arrs["A"]),
            _ptr(arrs["B"]), _ptr(arrs["C"]), _ptr(arrs["D"]), _ptr(arrs["z"]),
            _ptr(arrs["dt_bias"]), _ptr(arrs["init"]), _ptr(mask))
    return s, arrs, (S, T, H, P, G, N)


def forward(x, dt_raw, A, B, C, D=None, z=None, dt_bias=None, init=None, cu=None,
            heads=None, threads=0):
    """Sequential float64 forward.  Returns (y [T,H,P], final [S,H,P,N]).

    ``heads`` restricts the work to a subset of heads (other heads' outputs are 0).
    """
    s, keep, (S, T, H, P, G, N) = _make_in(x, dt_raw, A, B, C, D, z, dt_bias, init, cu, heads)
    y = np.zeros((T, H, P), dtype=np.float64)
    fin = np.zeros((S, H, P, N), dtype=np.float64)
    rc = _load().ssd_oracle_fwd(ctypes.byref(s), _ptr(y), _ptr(fin), int(threads))
    if rc != 0:
        raise RuntimeError("ssd_oracle_fwd failed with code %d" % rc)
    return y, fin


def backward(x, dt_raw, A, B, C, dy, D=None, z=None, dt_bias=None, init=None, dfinal=None,
             cu=None, heads=None, ckpt=128, threads=0):
    """Exact adjoint of :func:`forward` for L = sum(dy*y) + sum(dfinal*final).

    Returns a dict with dx, ddt_raw, dA, dB, dC and, when the matching input is
    given, dD, dz, ddt_bias, dinit.  With ``heads``, dB/dC only hold the listed
    heads' contributions.
    """
    s, keep, (S, T, H, P, G, N) = _make_in(x, dt_raw, A, B, C, D, z, dt_bias, init, cu, heads)
    dy = _f64(dy)
    dfinal = _f64(dfinal)
    out = dict(
        dx=np.zeros((T, H, P)), ddt_raw=np.zeros((T, H)), dA=np.zeros(H),
        dB=np.zeros((T, G, N)), dC=np.zeros((T, G, N)), dD=np.zeros(H),
        dz=np.zeros((T, H, P)), ddt_bias=np.zeros(H), dinit=np.zeros((S, H, P, N)),
    )
    rc = _load().ssd_oracle_bwd(
        ctypes.byref(s), _ptr(dy), _ptr(dfinal), _ptr(out["dx"]), _ptr(out["ddt_raw"]),
        _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dz"]),
        _ptr(out["ddt_bias"]), _ptr(out["dinit"]), int(ckpt), int(threads))
    if rc != 0:
        raise RuntimeError("ssd_oracle_bwd failed with code %d" % rc)
    if D is None:
        del out["dD"]
    if z is None:
        del out["dz"]
    if dt_bias is None:
        del out["ddt_bias"]
    if init is None:
        del out["dinit"]
    return out
