"""The C-ABI library without a GPU: it builds, loads, exports every entry point the public
header declares, and rejects bad arguments before touching CUDA (every check here
returns before the first CUDA runtime call, so no device is needed)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

OK, INVALID, UNSUPPORTED = 0, 1, 2
BAD_PTR = 0x1000        # never dereferenced: every call below fails validation first
BAD_PTR2 = 0x2000
MISALIGNED = 0x1008


@pytest.fixture(scope="module")
def lib():
    from rmsnorm_fwd_02_gb300 import build as B
    B.build()
    from rmsnorm_fwd_02_gb300 import _native as N
    return N.lib()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b((?:rmsnorm|layernorm)_train_\w+)\s*\(",
                                text, re.M)
    return names


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("rmsnorm_train_fwd", "rmsnorm_train_bwd",
                 "rmsnorm_train_bwd_workspace_bytes", "rmsnorm_train_status_str",
                 "rmsnorm_train_device_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from rmsnorm_fwd_02_gb300 import _native as N
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in N.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    from rmsnorm_fwd_02_gb300 import _native as N
    for st in range(0, 7):
        assert isinstance(N.status_str(st), str) and N.status_str(st)
    assert N.status_str(0) == "ok"


def fwd(lib, x=BAD_PTR, res=None, w=BAD_PTR, wd=0, y=BAD_PTR2, h=None, rstd=BAD_PTR2,
        T=4, nh=1, H=64, s_tok=64, s_head=64, eps=1e-6):
    return lib.rmsnorm_train_fwd(x, res, w, wd, y, h, rstd, T, nh, H, s_tok, s_head, eps,
                                 None)


def bwd(lib, x=BAD_PTR, dy=BAD_PTR, dh=None, rstd=BAD_PTR2, w=BAD_PTR, wd=0, dx=BAD_PTR2,
        dw=BAD_PTR2, ws=BAD_PTR, wsb=1 << 20, T=4, nh=1, H=64, s_tok=64, s_head=64, det=1):
    return lib.rmsnorm_train_bwd(x, dy, dh, rstd, w, wd, dx, dw, ws, wsb, T, nh, H, s_tok,
                                 s_head, det, None)


@pytest.mark.parametrize("kw,want", [
    (dict(H=60), INVALID),                   # H not a multiple of 8
    (dict(H=0), INVALID),
    (dict(H=8200, s_tok=8200), UNSUPPORTED),  # above the largest width
    (dict(T=-1), INVALID),
    (dict(nh=0), INVALID),
    (dict(x=None), INVALID),
    (dict(w=None), INVALID),
    (dict(y=None), INVALID),
    (dict(rstd=None), INVALID),
    (dict(x=MISALIGNED), INVALID),
    (dict(y=MISALIGNED), INVALID),
    (dict(wd=2), INVALID),
    (dict(res=BAD_PTR), INVALID),            # residual without h_out
    (dict(h=BAD_PTR2), INVALID),             # h_out without residual
    (dict(s_tok=60), INVALID),               # stride not a multiple of 8 elements
    (dict(nh=2, s_head=12), INVALID),
    (dict(eps=-1.0), INVALID),
    (dict(eps=float("nan")), INVALID),
    (dict(eps=float("inf")), INVALID),
    (dict(T=1 << 20, nh=4096), UNSUPPORTED),  # T*nh >= 2^31
    (dict(T=0), OK),                         # empty: nothing to do, no CUDA call
])
def test_fwd_rejects_before_any_cuda_call(lib, kw, want):
    assert fwd(lib, **kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(H=12), INVALID),
    (dict(det=2), INVALID),
    (dict(det=-1), INVALID),
    (dict(x=None), INVALID),
    (dict(dy=None), INVALID),
    (dict(rstd=None), INVALID),
    (dict(w=None), INVALID),
    (dict(dx=None), INVALID),
    (dict(dw=None), INVALID),
    (dict(dh=MISALIGNED), INVALID),
    (dict(ws=MISALIGNED), INVALID),
    (dict(rstd=BAD_PTR2 + 2), INVALID),
    (dict(wd=5), INVALID),
    (dict(H=16384, s_tok=16384), UNSUPPORTED),
])
def test_bwd_rejects_before_any_cuda_call(lib, kw, want):
    assert bwd(lib, **kw) == want


def test_deterministic_workspace_size_depends_on_shape_only(lib):
    f = lib.rmsnorm_train_bwd_workspace_bytes
    # up to 256 rows the backward runs in one launch without a workspace
    assert f(1, 1, 4096, 1) == 0
    assert f(256, 1, 4096, 1) == 0
    assert f(64, 4, 256, 1) == 0
    # H = 4096: one CTA an SM -> at most 152 partials of 2*H floats; a CTA takes at least
    # one stage (3 rows without dh, 2 with: the larger need, 2 rows, sets the size)
    assert f(65536, 1, 4096, 1) == 152 * 2 * 4096 * 4
    assert f(257, 1, 4096, 1) == 129 * 2 * 4096 * 4
    # H = 6144: 384 consumers, one CTA an SM -> at most 152
    assert f(65536, 1, 6144, 1) == 152 * 2 * 6144 * 4
    # H = 256 (the tensor-memory class): 64 eight-lane groups without dh, 32 with (four
    # stages; 32 rows a stage sets the size), one CTA an SM -> at most 152
    assert f(300, 1, 256, 1) == 10 * 2 * 256 * 4
    assert f(321, 1, 256, 1) == 11 * 2 * 256 * 4
    assert f(65536, 24, 256, 1) == 152 * 2 * 256 * 4
    # H = 8192: 4-vector threads, one CTA an SM
    assert f(131072, 1, 8192, 1) == 152 * 2 * 8192 * 4
    assert f(0, 1, 4096, 1) == 0
    assert f(10, 1, 12, 1) == 0       # invalid width


def test_package_import_needs_no_gpu():
    import rmsnorm_fwd_02_gb300 as R
    assert callable(R.rmsnorm_fwd) and callable(R.rmsnorm_train)


SMEM_PER_SM = 228 * 1024      # GB300 shared memory per SM, of which 1 KB per CTA is reserved
SMEM_PER_CTA = 227 * 1024


@pytest.mark.parametrize("op", [0, 1, 2, 3, 4, 5],
                         ids=["fwd", "fwd_res", "bwd", "bwd_dh", "bwd_nd", "bwd_nd_dh"])
def test_launch_plan_fits_its_kernel_build_at_every_width(lib, op):
    # Every supported width: the CTA fits the launch bounds of the kernel build it selects,
    # the ring and barriers fit shared memory at the build's CTAs per SM, the row groups
    # cover the row, and (backward) the ring can hold the end-of-kernel dw combine buffer.
    from rmsnorm_fwd_02_gb300 import _native as N
    tensors = {0: 1, 1: 2, 2: 2, 3: 3, 4: 2, 5: 3}[op]
    for H in range(8, 8193, 8):
        p = N.rmsnorm_train_launch_plan(H, op)
        ctx = f"H={H} {p}"
        assert p["threads"] == p["groups"] * p["group_threads"] + 32, ctx  # + producer warp
        assert p["threads"] % 32 == 0, ctx
        assert p["threads"] <= p["class_max_threads"], ctx
        assert p["smem"] <= SMEM_PER_CTA, ctx
        assert p["class_blocks_per_sm"] * (p["smem"] + 1024) <= SMEM_PER_SM, ctx
        assert p["stages"] >= 2, ctx
        assert p["group_threads"] * p["vpt"] * 8 >= H, ctx
        assert p["group_threads"] in (8, 16) or p["group_threads"] % 32 == 0, ctx
        if p["group_threads"] >= 32:
            assert p["groups"] <= 16, ctx          # reduction slots
        ring = p["stages"] * tensors * p["groups"] * H * 2
        if op >= 2:
            assert ring >= 8 * p["groups"] * H, ctx
            assert p["vpt"] in (1, 2, 3, 4), ctx
            if p["vpt"] == 3:
                assert p["cls"] in (1, 3), ctx  # 3-vector rows: the multi-group builds only
            if p["cls"] == 3:
                # the tensor-memory class: 608 consumers at most, whole warps, and each
                # thread's 16 columns a vector, four warps a lane quadrant, in 512 columns
                assert p["class_max_threads"] == 640, ctx
                warps = (p["threads"] - 32) // 32
                assert (p["threads"] - 32) % 32 == 0, ctx
                assert -(-warps // 4) * 16 * p["vpt"] <= 512, ctx
                assert p["stages"] >= 3, ctx
        else:
            if p["cls"] == 1:
                assert p["vpt"] in (2, 3, 4, 6), ctx   # the one-CTA forward's builds
                assert p["group_threads"] % 32 == 0, ctx
            else:
                assert p["vpt"] in (1, 2, 3, 4), ctx   # the two-CTA forward's builds


def test_launch_plan_rejects_bad_arguments(lib):
    out = (C.c_int64 * 9)()
    assert lib.rmsnorm_train_launch_plan(4096, 6, out, 9) == INVALID
    assert lib.rmsnorm_train_launch_plan(4096, -1, out, 9) == INVALID
    assert lib.rmsnorm_train_launch_plan(4100, 0, out, 9) == INVALID
    assert lib.rmsnorm_train_launch_plan(0, 0, out, 9) == INVALID
    assert lib.rmsnorm_train_launch_plan(8200, 0, out, 9) == UNSUPPORTED
    assert lib.rmsnorm_train_launch_plan(4096, 0, None, 9) == INVALID
    assert lib.rmsnorm_train_launch_plan(4096, 0, out, -1) == INVALID
    assert lib.rmsnorm_train_launch_plan(4096, 0, out, 0) == OK


def test_deterministic_workspace_covers_both_dh_plans(lib):
    # The backward's launch shape may differ with and without dh (the workspace query has
    # no dh argument): the size must cover the larger deterministic partition, which is
    # min(ceil(R / groups), 152 * CTAs an SM) partials of 2*H floats (a CTA takes at least
    # one stage of rows).
    from rmsnorm_fwd_02_gb300 import _native as N
    for H in (256, 768, 1536, 4096, 5120, 5632, 6144, 7168, 8192):
        for T in (1, 96, 700, 65536):
            need = 0
            if T <= 256:                       # one-launch path: no workspace
                assert lib.rmsnorm_train_bwd_workspace_bytes(T, 1, H, 1) == 0, (H, T)
                continue
            for op in (2, 3):
                p = N.rmsnorm_train_launch_plan(H, op)
                P = min(-(-T // p["groups"]), 152 * p["class_blocks_per_sm"])
                need = max(need, P * 2 * H * 4)
            assert lib.rmsnorm_train_bwd_workspace_bytes(T, 1, H, 1) == need, (H, T)


def test_nondeterministic_workspace_is_row_counter_and_partials(lib):
    # non-deterministic: a 16-byte row counter before the deterministic mode's partials;
    # no device query needed
    f = lib.rmsnorm_train_bwd_workspace_bytes
    for H in (8, 256, 1024, 1536, 4096, 6144, 8192):
        assert f(256, 1, H, 0) == 0
        for T in (257, 4096, 131072):
            assert f(T, 1, H, 0) == 16 + f(T, 1, H, 1), (H, T)
    assert f(65536, 24, 256, 0) == 16 + 152 * 2 * 256 * 4
    assert f(0, 1, 4096, 0) == 0


@pytest.mark.parametrize("dh", [False, True], ids=["plain", "dh"])
def test_both_modes_share_one_plan_at_every_width(lib, dh):
    # one row-pass program on one launch shape for both modes: dx is bit-identical across
    # them because every row is reduced the same way
    from rmsnorm_fwd_02_gb300 import _native as N
    for H in range(8, 8193, 8):
        a = N.rmsnorm_train_launch_plan(H, 3 if dh else 2)
        b = N.rmsnorm_train_launch_plan(H, 5 if dh else 4)
        assert a == b, (H, a, b)


@pytest.mark.parametrize("op", [2, 3], ids=["bwd", "bwd_dh"])
def test_backward_plan_counts_the_chunk_slots(lib, op):
    # the row pass keeps each stage's first and end row in shared memory (two words a
    # stage, rounded to 16 bytes): the plan's shared memory counts them
    from rmsnorm_fwd_02_gb300 import _native as N
    for H in range(8, 8193, 8):
        p = N.rmsnorm_train_launch_plan(H, op)
        tensors = 3 if op == 3 else 2
        ring = p["stages"] * tensors * p["groups"] * H * 2
        assert p["smem"] >= ring + 4 * ((2 * p["stages"] + 3) // 4 * 4), (H, p)


def test_noalloc_scratch_covers_every_supported_shape(lib):
    # rmsnorm_train_bwd_noalloc keeps its workspace in a 16 MiB array: the partition is at
    # most 152 x (CTAs an SM) partials of 2*H floats (+ a 16-byte counter in the
    # non-deterministic mode), so no supported shape reaches the limit
    f = lib.rmsnorm_train_bwd_workspace_bytes
    for H in range(8, 8193, 8):
        for det in (0, 1):
            assert f(1 << 20, 1, H, det) <= 16 << 20, (H, det)


def test_recompute_rejects_before_any_cuda_call(lib):
    f = lib.rmsnorm_train_bwd_recompute
    args = dict(x=BAD_PTR, dy=BAD_PTR, dh=None, w=BAD_PTR, wd=0, dx=BAD_PTR2, dw=BAD_PTR2,
                rs=BAD_PTR2, ws=None, wsb=0, T=300, nh=1, H=4096, st=4096, sh=4096, eps=1e-6,
                det=1)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["x"], a["dy"], a["dh"], a["w"], a["wd"], a["dx"], a["dw"], a["rs"], a["ws"],
                 a["wsb"], a["T"], a["nh"], a["H"], a["st"], a["sh"], a["eps"], a["det"], None)

    assert call(rs=None) == INVALID                  # rstd_out is required
    assert call(rs=BAD_PTR2 + 2) == INVALID          # and 4-byte aligned
    assert call(eps=float("nan")) == INVALID
    assert call(eps=-1.0) == INVALID
    assert call(H=12, st=12, sh=12) == INVALID
    assert call(x=None) == INVALID
    assert call(det=3) == INVALID
