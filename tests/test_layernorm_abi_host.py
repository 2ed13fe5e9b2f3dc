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
    (dict(H=8200), UNSUPPORTED),             # past 8192 the width must split into 16-byte halves
    (dict(H=16400), UNSUPPORTED),
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
    (dict(H=16400), UNSUPPORTED),
    (dict(H=12296), UNSUPPORTED),            # a multiple of 8, not of 16, past 8192
    (dict(H=16384, x=None), INVALID),        # the widest width is supported: the checks go on
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


def _widths():
    # every supported width: multiples of 8 up to 8192, multiples of 16 up to 16384
    return list(range(8, 8193, 8)) + list(range(8208, 16385, 16))


@pytest.mark.parametrize("op", [LN_FWD, LN_BWD], ids=["fwd", "bwd"])
def test_layernorm_plan_fits_its_kernel_build_at_every_width(lib, op):
    tensors = 1 if op == LN_FWD else 2
    for H in _widths():
        p = _plan(H, op)
        ctx = f"H={H} {p}"
        pair = p["cluster_ctas"] == 2
        assert p["cluster_ctas"] == (2 if H > 8192 else 1), ctx
        Hc = H // 2 if pair else H                     # the columns one CTA owns
        assert p["threads"] == p["groups"] * p["group_threads"] + 32, ctx
        assert p["threads"] % 32 == 0, ctx
        assert p["threads"] <= p["class_max_threads"], ctx
        assert p["class_blocks_per_sm"] == 1, ctx
        assert p["smem"] <= SMEM_PER_CTA, ctx
        assert p["stages"] >= 2, ctx
        assert p["group_threads"] * p["vpt"] * 8 >= Hc, ctx
        assert p["group_threads"] in (8, 16) or p["group_threads"] % 32 == 0, ctx
        if p["group_threads"] >= 32:
            assert p["groups"] <= 16, ctx             # reduction slots and warp tables
        if pair:
            assert p["group_threads"] >= 32, ctx      # a pair exchanges whole warps' partials
            assert (Hc * 2) % 16 == 0, ctx            # 16-byte half-rows for the bulk copies
            warps_both = 2 * p["group_threads"] // 32
            assert 2 * warps_both <= 64, ctx          # two slot floats a warp of the pair
        if op == LN_FWD:
            if pair:
                assert (p["cls"], p["vpt"]) == (3, 4) and p["class_max_threads"] == 640, ctx
            else:
                assert p["cls"] == 0 and p["vpt"] in (1, 2, 4), ctx
                assert p["class_max_threads"] == 640, ctx
        else:
            assert (p["cls"], p["vpt"]) in ((1, 1), (1, 2), (2, 3), (5, 2), (5, 3), (5, 4)), ctx
            assert p["class_max_threads"] == {1: 512, 2: 384, 5: 640}[p["cls"]], ctx
            if pair:
                assert p["cls"] != 5 or p["vpt"] == 4, ctx   # the one pair build of it
            if p["cls"] == 5:
                # the tensor-memory class: whole consumer warps, 32 columns of a thread's
                # lane a column vector, four warps a lane quadrant, within 512 columns
                cons = p["threads"] - 32
                assert cons % 32 == 0, ctx
                assert -(-(cons // 32) // 4) * 32 * p["vpt"] <= 512, ctx
                assert p["stages"] >= 3, ctx
            ring = p["stages"] * tensors * p["groups"] * Hc * 2
            assert ring >= 8 * p["groups"] * Hc, ctx   # the end-of-kernel combine buffer


def test_layernorm_plan_rejects_bad_arguments(lib):
    out = (C.c_int64 * 10)()
    assert lib.layernorm_train_launch_plan(4096, 2, out, 10) == INVALID
    assert lib.layernorm_train_launch_plan(4100, 0, out, 10) == INVALID
    assert lib.layernorm_train_launch_plan(8200, 0, out, 10) == UNSUPPORTED
    assert lib.layernorm_train_launch_plan(16400, 1, out, 10) == UNSUPPORTED
    assert lib.layernorm_train_launch_plan(4096, 0, None, 10) == INVALID
    assert lib.layernorm_train_launch_plan(4096, 1, out, 0) == OK
    assert lib.layernorm_train_launch_plan(16384, 1, out, 10) == OK and out[9] == 2


def test_layernorm_deterministic_workspace_depends_on_shape_only(lib):
    # P row chunks of one CTA (at most 152) or of a CTA pair (at most 76), each writing a
    # partial row of 4*H floats (dw and db, hi and lo)
    f = lib.layernorm_train_bwd_workspace_bytes
    for H in (8, 256, 1000, 3584, 4096, 7680, 8192, 8208, 12288, 16384):
        p = _plan(H, LN_BWD)
        cap = 152 // p["cluster_ctas"]
        for R in (1, 7, 300, 8192, 65536):
            P = min(-(-R // p["groups"]), cap)
            assert f(R, H, 1) == P * 4 * H * 4, (H, R)
    assert f(0, 4096, 1) == 0
    assert f(10, 12, 1) == 0
    assert f(10, 16400, 1) == 0
