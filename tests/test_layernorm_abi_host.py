"""The LayerNorm entry points of the C-ABI library without a GPU: declared, exported and
bound; bad arguments rejected before the first CUDA runtime call; launch plans that fit
their kernel builds at every width; a deterministic workspace that depends on the shape
only.  (LayerNorm with weight and bias, the normalization benchmarked beside RMSNorm in
ROCm TransformerEngine PR #478's normalization tables.)"""
import ctypes as C

import pytest

from test_abi_host import BAD_PTR, BAD_PTR2, INVALID, MISALIGNED, OK, UNSUPPORTED, \
    declared_functions, lib  # noqa: F401  (lib: the module fixture)

SMEM_PER_CTA = 227 * 1024
LN_FWD, LN_BWD = 0, 1


def test_header_declares_layernorm_entry_points():
    names = declared_functions()
    for want in ("layernorm_train_fwd", "layernorm_train_bwd",
                 "layernorm_train_bwd_workspace_bytes", "layernorm_train_launch_plan",
                 "layernorm_train_device_error"):
        assert want in names


def fwd(lib, x=BAD_PTR, w=BAD_PTR, b=BAD_PTR, wd=0, y=BAD_PTR2, mean=BAD_PTR2,
        rstd=BAD_PTR2, R=4, H=64, eps=1e-5):
    return lib.layernorm_train_fwd(x, w, b, wd, y, mean, rstd, R, H, eps, None)


def bwd(lib, x=BAD_PTR, dy=BAD_PTR, mean=BAD_PTR2, rstd=BAD_PTR2, w=BAD_PTR, wd=0,
        dx=BAD_PTR2, dw=BAD_PTR2, db=BAD_PTR2, ws=BAD_PTR, wsb=1 << 20, R=4, H=64, det=1):
    return lib.layernorm_train_bwd(x, dy, mean, rstd, w, wd, dx, dw, db, ws, wsb, R, H, det,
                                   None)


@pytest.mark.parametrize("kw,want", [
    (dict(H=60), INVALID),
    (dict(H=0), INVALID),
    (dict(H=8200), UNSUPPORTED),
    (dict(R=-1), INVALID),
    (dict(R=1 << 31), UNSUPPORTED),
    (dict(x=None), INVALID),
    (dict(w=None), INVALID),
    (dict(b=None), INVALID),
    (dict(y=None), INVALID),
    (dict(mean=None), INVALID),
    (dict(rstd=None), INVALID),
    (dict(x=MISALIGNED), INVALID),
    (dict(b=MISALIGNED), INVALID),
    (dict(y=MISALIGNED), INVALID),
    (dict(mean=BAD_PTR2 + 2), INVALID),
    (dict(wd=2), INVALID),
    (dict(eps=-1.0), INVALID),
    (dict(eps=float("nan")), INVALID),
    (dict(R=0), OK),                         # empty: nothing to do, no CUDA call
    (dict(R=0, x=None, y=None, mean=None, rstd=None), OK),   # no rows: row tensors unused
    (dict(R=0, w=None), INVALID),
])
def test_layernorm_fwd_rejects_before_any_cuda_call(lib, kw, want):
    assert fwd(lib, **kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(H=12), INVALID),
    (dict(H=16384), UNSUPPORTED),
    (dict(det=2), INVALID),
    (dict(x=None), INVALID),
    (dict(dy=None), INVALID),
    (dict(mean=None), INVALID),
    (dict(rstd=None), INVALID),
    (dict(w=None), INVALID),
    (dict(dx=None), INVALID),
    (dict(dw=None), INVALID),
    (dict(db=None), INVALID),
    (dict(db=MISALIGNED), INVALID),
    (dict(ws=MISALIGNED), INVALID),
    (dict(rstd=BAD_PTR2 + 1), INVALID),
    (dict(wd=7), INVALID),
    (dict(R=0, db=None), INVALID),           # dw and db are written even with no rows
])
def test_layernorm_bwd_rejects_before_any_cuda_call(lib, kw, want):
    assert bwd(lib, **kw) == want


def _plan(H, op):
    from rmsnorm_fwd_02_gb300 import _native as N
    return N.layernorm_train_launch_plan(H, op)


@pytest.mark.parametrize("op", [LN_FWD, LN_BWD], ids=["fwd", "bwd"])
def test_layernorm_plan_fits_its_kernel_build_at_every_width(lib, op):
    tensors = 1 if op == LN_FWD else 2
    for H in range(8, 8193, 8):
        p = _plan(H, op)
        ctx = f"H={H} {p}"
        assert p["threads"] == p["groups"] * p["group_threads"] + 32, ctx
        assert p["threads"] % 32 == 0, ctx
        assert p["threads"] <= p["class_max_threads"], ctx
        assert p["class_blocks_per_sm"] == 1, ctx
        assert p["smem"] <= SMEM_PER_CTA, ctx
        assert p["stages"] >= 2, ctx
        assert p["group_threads"] * p["vpt"] * 8 >= H, ctx
        assert p["group_threads"] in (8, 16) or p["group_threads"] % 32 == 0, ctx
        if p["group_threads"] >= 32:
            assert p["groups"] <= 16, ctx             # reduction slots and warp tables
        if op == LN_FWD:
            assert p["cls"] == 0 and p["vpt"] in (1, 2, 4), ctx
            assert p["class_max_threads"] == 512, ctx
        else:
            assert (p["cls"], p["vpt"]) in ((1, 1), (1, 2), (2, 3)), ctx
            assert p["class_max_threads"] == (512 if p["cls"] == 1 else 384), ctx
            ring = p["stages"] * tensors * p["groups"] * H * 2
            assert ring >= 8 * p["groups"] * H, ctx     # the end-of-kernel combine buffer


def test_layernorm_plan_rejects_bad_arguments(lib):
    out = (C.c_int64 * 9)()
    assert lib.layernorm_train_launch_plan(4096, 2, out, 9) == INVALID
    assert lib.layernorm_train_launch_plan(4100, 0, out, 9) == INVALID
    assert lib.layernorm_train_launch_plan(8200, 0, out, 9) == UNSUPPORTED
    assert lib.layernorm_train_launch_plan(4096, 0, None, 9) == INVALID
    assert lib.layernorm_train_launch_plan(4096, 1, out, 0) == OK


def test_layernorm_deterministic_workspace_depends_on_shape_only(lib):
    f = lib.layernorm_train_bwd_workspace_bytes
    for H in (8, 256, 1000, 3584, 4096, 7680, 8192):
        G = _plan(H, LN_BWD)["groups"]
        for R in (1, 7, 300, 8192, 65536):
            P = min(-(-R // G), 152)
            assert f(R, H, 1) == P * 4 * H * 4, (H, R)
    assert f(0, 4096, 1) == 0
    assert f(10, 12, 1) == 0
    assert f(10, 16384, 1) == 0
