"""FP64 CPU oracle for RMSNorm training -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline (and its
reference arm) may import this package.  The product library never does, and it shares
no code with it.  The arithmetic lives in ``rmsnorm_oracle.c`` (plain C, IEEE double,
sequential loops); this module only moves numpy arrays in and out through ctypes.

The operation is the one flashinfer PR #8827 ("fix(cake_rmsnorm): sm_100a and sm_107a
dw-accuracy backward routes") states in its description: forward y = x*rstd*w with
rstd = 1/sqrt(mean(x^2)+eps), an optional fused residual add whose BF16 sum h_new is
written, and a backward returning dx and dw = sum over rows of dy*xhat; per-head views
address row (t, h) at t*s_tok + h*s_head.  Every function below says which part it covers.

Array conventions: BF16 tensors are numpy ``uint16`` bit patterns; FP32 weights are
``float32``; FP64 inputs (for gradient checks) are ``float64``.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from .build import build_oracle

_BF16, _F32, _F64 = 0, 1, 2
_libs: dict = {}


def _load(path: str | None = None):
    """Loads the oracle library (the default build, or another build of the same source
    at ``path``) and declares its C signatures."""
    path = path or build_oracle()
    lib = _libs.get(path)
    if lib is None:
        lib = C.CDLL(path)
        i64, i32, vp, dp = C.c_int64, C.c_int32, C.c_void_p, C.c_double
        lib.orc_f64_to_bf16_rne.restype = C.c_uint16
        lib.orc_f64_to_bf16_rne.argtypes = [dp]
        lib.orc_bf16_to_f64.restype = dp
        lib.orc_bf16_to_f64.argtypes = [C.c_uint16]
        lib.orc_round_bf16.restype = None
        lib.orc_round_bf16.argtypes = [vp, vp, i64]
        lib.orc_fwd.restype = None
        lib.orc_fwd.argtypes = [i64, i32, i32, i64, i64, vp, C.c_int, vp, C.c_int, vp,
                                C.c_int, dp, vp, i64, vp, vp, vp, vp]
        lib.orc_bwd_dx.restype = None
        lib.orc_bwd_dx.argtypes = [i64, i32, i32, i64, i64, vp, C.c_int, vp, C.c_int, vp,
                                   C.c_int, vp, vp, C.c_int, vp, i64, vp, vp]
        lib.orc_bwd_dw.restype = None
        lib.orc_bwd_dw.argtypes = [i64, i32, i32, i64, i64, vp, C.c_int, vp, C.c_int,
                                   vp, vp]
        _libs[path] = lib
    return lib


_active_path: str | None = None


def use_library(path: str | None) -> None:
    """Points this module at another build of ``rmsnorm_oracle.c`` (None: the default).
    Only the mutation tests use this, to show that the pins reject planted mistakes."""
    global _active_path
    _active_path = path


def _lib():
    return _load(_active_path)


def _kind(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return _BF16
    if a.dtype == np.float32:
        return _F32
    if a.dtype == np.float64:
        return _F64
    raise TypeError(f"unsupported oracle input dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a):
    return None if a is None else np.ascontiguousarray(a)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns to FP64 (a BF16 value is the top half of an
    FP32 value)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round FP64 values to BF16 (nearest, ties to even) in one step; returns bits.

    The PR's workload line fixes y, dx and h_new as BF16; rounding to nearest-even is the
    IEEE default that the comparison uses."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _lib().orc_round_bf16(_ptr(v), _ptr(out), v.size)
    return out


def fwd(x, w, eps, T, nh, H, s_tok, s_head, residual=None, rows=None, want_y=True):
    """Forward of the op (description of PR #8827: y (BF16) and rstd (FP32); fused
    residual add writing h_new = BF16(h + u)).

    ``x`` (and ``residual``) are flat arrays addressed through the view strides.
    Returns ``(y64 [n, H] or None, rstd64 [n], h_bits [n, H] or None)`` for the selected
    rows (all rows when ``rows`` is None)."""
    lib = _lib()
    x = _c(x)
    residual = _c(residual)
    w = _c(w)
    R = T * nh
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = R if rows_a is None else rows_a.size
    y = np.empty((n, H), np.float64) if want_y else None
    rstd = np.empty(n, np.float64)
    h = np.empty((n, H), np.uint16) if residual is not None else None
    scratch = np.empty(H, np.float64)
    lib.orc_fwd(T, nh, H, s_tok, s_head, _ptr(x), _kind(x), _ptr(residual),
                _kind(residual) if residual is not None else 0, _ptr(w), _kind(w),
                float(eps), _ptr(rows_a), n, _ptr(y), _ptr(rstd), _ptr(h), _ptr(scratch))
    return y, rstd, h


def bwd_dx(x, dy, r_all, w, T, nh, H, s_tok, s_head, dh=None, rows=None):
    """dx of the backward (PR #8827 description: the backward's BF16 input gradient) for
    the selected rows, with the rstd ``r_all`` (FP64, one per row) the backward is
    handed.  The residual form's combined gradient adds ``dh``.  Returns FP64 [n, H]."""
    lib = _lib()
    x, dy, dh, w = _c(x), _c(dy), _c(dh), _c(w)
    r_all = np.ascontiguousarray(r_all, dtype=np.float64)
    R = T * nh
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = R if rows_a is None else rows_a.size
    dx = np.empty((n, H), np.float64)
    scratch = np.empty(2 * H, np.float64)
    lib.orc_bwd_dx(T, nh, H, s_tok, s_head, _ptr(x), _kind(x), _ptr(dy), _kind(dy),
                   _ptr(dh), _kind(dh) if dh is not None else 0, _ptr(r_all), _ptr(w),
                   _kind(w), _ptr(rows_a), n, _ptr(dx), _ptr(scratch))
    return dx


def bwd_dw(x, dy, r_all, T, nh, H, s_tok, s_head):
    """dw of the backward (PR #8827 description: the FP32 weight gradient; PR #8849,
    changed windows: the accuracy budget is taken against an FP64 sum): the sum over
    every row, in row order, of dy * x * r.  Returns FP64 [H]."""
    lib = _lib()
    x, dy = _c(x), _c(dy)
    r_all = np.ascontiguousarray(r_all, dtype=np.float64)
    dw = np.empty(H, np.float64)
    lib.orc_bwd_dw(T, nh, H, s_tok, s_head, _ptr(x), _kind(x), _ptr(dy), _kind(dy),
                   _ptr(r_all), _ptr(dw))
    return dw
