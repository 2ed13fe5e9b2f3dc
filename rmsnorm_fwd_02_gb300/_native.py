"""ctypes binding of ``librmsnorm_train.so`` with the C ABI's names (include/rmsnorm_train.h
and include/layernorm_train.h).

Argument marshalling only: tensors become device pointers, the current torch stream
becomes the ``cudaStream_t``, sizes and strides are passed through, and a nonzero status
becomes an exception.  Every step of the computation runs in the CUDA library; there is
no fallback.  If the library is missing this module raises on first use.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librmsnorm_train.so")

RMSN_OK = 0
RMSN_W_BF16 = 0
RMSN_W_FP32 = 1

# every C entry point declared in include/rmsnorm_train.h, with its ctypes signature
_i64, _i32, _vp, _int, _f32, _size = (C.c_int64, C.c_int32, C.c_void_p, C.c_int, C.c_float,
                                      C.c_size_t)
SIGNATURES = {
    "rmsnorm_train_fwd": (_int, [_vp, _vp, _vp, _int, _vp, _vp, _vp, _i64, _i32, _i32, _i64,
                                 _i64, _f32, _vp]),
    "rmsnorm_train_bwd_workspace_bytes": (_size, [_i64, _i32, _i32, _int]),
    "rmsnorm_train_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _vp, _size, _i64,
                                 _i32, _i32, _i64, _i64, _int, _vp]),
    "rmsnorm_train_bwd_noalloc": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _i64, _i32,
                                         _i32, _i64, _i64, _int, _vp]),
    "rmsnorm_train_bwd_recompute": (_int, [_vp, _vp, _vp, _vp, _int, _vp, _vp, _vp, _vp, _size,
                                           _i64, _i32, _i32, _i64, _i64, _f32, _int, _vp]),
    "rmsnorm_train_status_str": (C.c_char_p, [_int]),
    "rmsnorm_train_device_error": (_int, [C.POINTER(C.c_uint), _int]),
    "rmsnorm_train_launch_plan": (_int, [_i32, _int, C.POINTER(C.c_int64), _int]),
    # include/layernorm_train.h
    "layernorm_train_fwd": (_int, [_vp, _vp, _vp, _int, _vp, _vp, _vp, _i64, _i32, _f32, _vp]),
    "layernorm_train_bwd_workspace_bytes": (_size, [_i64, _i32, _int]),
    "layernorm_train_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _vp, _vp, _size,
                                   _i64, _i32, _int, _vp]),
    "layernorm_train_launch_plan": (_int, [_i32, _int, C.POINTER(C.c_int64), _int]),
    "layernorm_train_device_error": (_int, [C.POINTER(C.c_uint), _int]),
}

PLAN_FWD, PLAN_FWD_RESIDUAL, PLAN_BWD, PLAN_BWD_DH, PLAN_BWD_ND, PLAN_BWD_ND_DH = 0, 1, 2, 3, 4, 5
LN_PLAN_FWD, LN_PLAN_BWD = 0, 1
PLAN_FIELDS = ("vpt", "group_threads", "groups", "stages", "threads", "smem", "cls",
               "class_max_threads", "class_blocks_per_sm")
LN_PLAN_FIELDS = PLAN_FIELDS + ("cluster_ctas",)

_lib = None


class RmsnError(RuntimeError):
    """A nonzero status from the CUDA library."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: status {status} ({status_str(status)})")
        self.status = status


def lib():
    """The loaded library.  Raises if it has not been built: there is no CPU path."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library {LIB_PATH} is missing; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_str(status: int) -> str:
    return lib().rmsnorm_train_status_str(status).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def rmsnorm_train_fwd(x, residual, w, w_dtype, y, h_out, rstd, T, nh, H, s_tok, s_head,
                      eps, stream=None):
    st = lib().rmsnorm_train_fwd(_ptr(x), _ptr(residual), _ptr(w), w_dtype, _ptr(y),
                                 _ptr(h_out), _ptr(rstd), T, nh, H, s_tok, s_head, eps,
                                 _stream(stream))
    if st != RMSN_OK:
        raise RmsnError("rmsnorm_train_fwd", st)


def rmsnorm_train_bwd_workspace_bytes(T, nh, H, deterministic):
    return int(lib().rmsnorm_train_bwd_workspace_bytes(T, nh, H, int(deterministic)))


def rmsnorm_train_bwd(x, dy, dh, rstd, w, w_dtype, dx, dw, workspace, workspace_bytes, T, nh,
                      H, s_tok, s_head, deterministic, stream=None):
    st = lib().rmsnorm_train_bwd(_ptr(x), _ptr(dy), _ptr(dh), _ptr(rstd), _ptr(w), w_dtype,
                                 _ptr(dx), _ptr(dw), _ptr(workspace), workspace_bytes, T, nh,
                                 H, s_tok, s_head, int(deterministic), _stream(stream))
    if st != RMSN_OK:
        raise RmsnError("rmsnorm_train_bwd", st)


def rmsnorm_train_bwd_recompute(x, dy, dh, w, w_dtype, dx, dw, rstd_out, workspace,
                                workspace_bytes, T, nh, H, s_tok, s_head, eps, deterministic,
                                stream=None):
    st = lib().rmsnorm_train_bwd_recompute(_ptr(x), _ptr(dy), _ptr(dh), _ptr(w), w_dtype,
                                           _ptr(dx), _ptr(dw), _ptr(rstd_out), _ptr(workspace),
                                           workspace_bytes, T, nh, H, s_tok, s_head, eps,
                                           int(deterministic), _stream(stream))
    if st != RMSN_OK:
        raise RmsnError("rmsnorm_train_bwd_recompute", st)


def rmsnorm_train_bwd_noalloc(x, dy, dh, rstd, w, w_dtype, dx, dw, T, nh, H, s_tok, s_head,
                              deterministic, stream=None):
    st = lib().rmsnorm_train_bwd_noalloc(_ptr(x), _ptr(dy), _ptr(dh), _ptr(rstd), _ptr(w),
                                         w_dtype, _ptr(dx), _ptr(dw), T, nh, H, s_tok, s_head,
                                         int(deterministic), _stream(stream))
    if st != RMSN_OK:
        raise RmsnError("rmsnorm_train_bwd_noalloc", st)


def rmsnorm_train_status_str(status):
    return status_str(status)


def rmsnorm_train_device_error(reset=True):
    flags = C.c_uint(0)
    st = lib().rmsnorm_train_device_error(C.byref(flags), int(reset))
    if st != RMSN_OK:
        raise RmsnError("rmsnorm_train_device_error", st)
    return int(flags.value)


def rmsnorm_train_launch_plan(H, op):
    """The library's launch plan for one op (PLAN_*) at width H, as a dict."""
    out = (C.c_int64 * len(PLAN_FIELDS))()
    st = lib().rmsnorm_train_launch_plan(H, op, out, len(PLAN_FIELDS))
    if st != RMSN_OK:
        raise RmsnError("rmsnorm_train_launch_plan", st)
    return dict(zip(PLAN_FIELDS, (int(v) for v in out)))


# ---- LayerNorm (include/layernorm_train.h) ----------------------------------------------

def layernorm_train_fwd(x, w, b, wb_dtype, y, mean, rstd, R, H, eps, stream=None):
    st = lib().layernorm_train_fwd(_ptr(x), _ptr(w), _ptr(b), wb_dtype, _ptr(y), _ptr(mean),
                                   _ptr(rstd), R, H, eps, _stream(stream))
    if st != RMSN_OK:
        raise RmsnError("layernorm_train_fwd", st)


def layernorm_train_bwd_workspace_bytes(R, H, deterministic):
    return int(lib().layernorm_train_bwd_workspace_bytes(R, H, int(deterministic)))


def layernorm_train_bwd(x, dy, mean, rstd, w, wb_dtype, dx, dw, db, workspace, workspace_bytes,
                        R, H, deterministic, stream=None):
    st = lib().layernorm_train_bwd(_ptr(x), _ptr(dy), _ptr(mean), _ptr(rstd), _ptr(w), wb_dtype,
                                   _ptr(dx), _ptr(dw), _ptr(db), _ptr(workspace),
                                   workspace_bytes, R, H, int(deterministic), _stream(stream))
    if st != RMSN_OK:
        raise RmsnError("layernorm_train_bwd", st)


def layernorm_train_launch_plan(H, op):
    """The library's LayerNorm launch plan for op LN_PLAN_FWD / LN_PLAN_BWD, as a dict."""
    out = (C.c_int64 * len(LN_PLAN_FIELDS))()
    st = lib().layernorm_train_launch_plan(H, op, out, len(LN_PLAN_FIELDS))
    if st != RMSN_OK:
        raise RmsnError("layernorm_train_launch_plan", st)
    return dict(zip(LN_PLAN_FIELDS, (int(v) for v in out)))


def layernorm_train_device_error(reset=True):
    flags = C.c_uint(0)
    st = lib().layernorm_train_device_error(C.byref(flags), int(reset))
    if st != RMSN_OK:
        raise RmsnError("layernorm_train_device_error", st)
    return int(flags.value)
