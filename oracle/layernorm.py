"""FP64 CPU oracle for LayerNorm training -- TEST INFRASTRUCTURE.

The arithmetic lives in ``layernorm_oracle.c`` (plain C, IEEE double, sequential loops);
this module moves numpy arrays in and out through ctypes.  LayerNorm is the normalization
beside RMSNorm in the ROCm TransformerEngine PR #478 microbenchmark tables; the pages print
no formula for it, so the oracle is the textbook definition with weight and bias:
y = (x - mean) * rstd * w + b, rstd = 1/sqrt(var + eps) with a two-pass variance, and the
backward dx = rstd * (g - mean(g) - xhat * mean(g * xhat)), dw = sum dy * xhat, db = sum dy.

Arrays: rows contiguous [R, H]; BF16 as numpy ``uint16`` bit patterns, FP32 ``float32``,
FP64 ``float64`` (for gradient checks).
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from .build import build_layernorm_oracle

_libs: dict = {}
_active_path: str | None = None


def use_library(path: str | None) -> None:
    """Points this module at another build of ``layernorm_oracle.c`` (None: the default);
    the mutation tests use it to show that the pins reject planted mistakes."""
    global _active_path
    _active_path = path


def _lib():
    path = _active_path or build_layernorm_oracle()
    lib = _libs.get(path)
    if lib is None:
        lib = C.CDLL(path)
        i64, i32, vp, dp, ci = C.c_int64, C.c_int32, C.c_void_p, C.c_double, C.c_int
        lib.ln_fwd.restype = None
        lib.ln_fwd.argtypes = [i64, i32, vp, ci, vp, ci, vp, ci, dp, vp, vp, vp]
        lib.ln_bwd_dx.restype = None
        lib.ln_bwd_dx.argtypes = [i64, i32, vp, ci, vp, ci, vp, vp, vp, ci, vp, vp]
        lib.ln_bwd_dw_db.restype = None
        lib.ln_bwd_dw_db.argtypes = [i64, i32, vp, ci, vp, ci, vp, vp, vp, vp]
        _libs[path] = lib
    return lib


def _kind(a: np.ndarray) -> int:
    return {np.dtype(np.uint16): 0, np.dtype(np.float32): 1, np.dtype(np.float64): 2}[a.dtype]


def fwd(x, w, b, eps, R, H, want_y=True):
    """Forward over R contiguous rows: returns (y64 [R, H] or None, mean [R], rstd [R])."""
    x, w, b = (np.ascontiguousarray(a) for a in (x, w, b))
    y = np.empty((R, H), np.float64) if want_y else None
    mean = np.empty(R, np.float64)
    rstd = np.empty(R, np.float64)
    _lib().ln_fwd(R, H, x.ctypes.data, _kind(x), w.ctypes.data, _kind(w), b.ctypes.data,
                  _kind(b), float(eps), None if y is None else y.ctypes.data,
                  mean.ctypes.data, rstd.ctypes.data)
    return y, mean, rstd


def bwd_dx(x, dy, mean, rstd, w, R, H):
    """dx (FP64 [R, H]) with the mean and rstd the backward is handed."""
    x, dy, w = (np.ascontiguousarray(a) for a in (x, dy, w))
    mean = np.ascontiguousarray(mean, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    dx = np.empty((R, H), np.float64)
    scratch = np.empty(2 * H, np.float64)
    _lib().ln_bwd_dx(R, H, x.ctypes.data, _kind(x), dy.ctypes.data, _kind(dy),
                     mean.ctypes.data, rstd.ctypes.data, w.ctypes.data, _kind(w),
                     dx.ctypes.data, scratch.ctypes.data)
    return dx


def bwd_dw_db(x, dy, mean, rstd, R, H):
    """dw and db (FP64 [H] each), summed over the rows in increasing order."""
    x, dy = (np.ascontiguousarray(a) for a in (x, dy))
    mean = np.ascontiguousarray(mean, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    dw = np.empty(H, np.float64)
    db = np.empty(H, np.float64)
    _lib().ln_bwd_dw_db(R, H, x.ctypes.data, _kind(x), dy.ctypes.data, _kind(dy),
                        mean.ctypes.data, rstd.ctypes.data, dw.ctypes.data, db.ctypes.data)
    return dw, db
