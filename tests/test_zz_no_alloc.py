"""rmsnorm_train_bwd_noalloc: the backward for callers that cannot allocate device memory
where they call it (e.g. a plugin's enqueue callback in a runtime that forbids
allocation there).  It keeps its dw partials in a device array built into the library
instead of a caller workspace.

Called through the C ABI, it must give what rmsnorm_train_bwd gives with a workspace:
dx within the 1-BF16-ulp gate and dw within the per-element budget of each other (in
fact the same kernels run, so dx's bits match, and dw's in the deterministic mode).  Two calls in a row on different shapes
check that the shared array's leftover contents from the previous call never leak into
the next one.  This file sorts last so a stop-at-first-failure run has already run
every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from rmsnorm_fwd_02_gb300 import _native as N
from rmsnorm_fwd_02_gb300 import synth
import parity

pytestmark = pytest.mark.gpu


def _with_workspace(dc, rstd, det):
    c = dc.c
    return parity.gpu_bwd(dc, dc.x, c.s_tok, c.s_head, rstd, det)


def _without_workspace(dc, rstd, det):
    c = dc.c
    dx = torch.empty(c.R * c.H, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((c.H,), float("nan"), dtype=torch.float32, device="cuda")
    N.rmsnorm_train_bwd_noalloc(dc.x, dc.dy, None, rstd, dc.w, parity.wdtype(c), dx, dw,
                                c.T, c.nh, c.H, c.s_tok, c.s_head, det)
    return dx, dw


def _agree(a, b, det):
    (dx_a, dw_a), (dx_b, dw_b) = a, b
    ba, bb = parity.bits_of(dx_a), parity.bits_of(dx_b)
    assert np.abs(parity.ordinal(ba) - parity.ordinal(bb)).max() <= 1
    wa, wb = dw_a.cpu().numpy().astype(np.float64), dw_b.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(wa - wb) <= parity.DW_ATOL + parity.DW_RTOL * np.abs(wa))
    # the same kernels run: dx is identical; so is dw in the deterministic mode (the
    # non-deterministic one hands rows to its CTAs as they come, so dw's last bits vary)
    assert np.array_equal(ba, bb)
    if det:
        assert np.array_equal(wa, wb)


@pytest.mark.parametrize("det", [1, 0])
def test_noalloc_matches_workspace_backward_on_two_calls_in_a_row(det):
    cases = [synth.plain(4096, seed=3), synth.stress(65536, 5120, seed=4),
             synth.heads_strided(512, seed=5)]
    for c in cases:
        dc = parity.DeviceCase(c)
        _, rstd, _ = parity.gpu_fwd(dc, False)
        ref = _with_workspace(dc, rstd, det)
        first = _without_workspace(dc, rstd, det)
        torch.cuda.synchronize()
        _agree(ref, first, det)
    # and back to the first shape: the array now holds the last shape's partials
    c = cases[0]
    dc = parity.DeviceCase(c)
    _, rstd, _ = parity.gpu_fwd(dc, False)
    ref = _with_workspace(dc, rstd, det)
    again = _without_workspace(dc, rstd, det)
    torch.cuda.synchronize()
    _agree(ref, again, det)
    assert N.rmsnorm_train_device_error(reset=True) == 0


def test_noalloc_scratch_limit_is_reported():
    # the largest partition this library plans fits the built-in 16 MiB
    for T, H, det in [(131072, 8192, 1), (65536, 4096, 1), (131072, 6144, 0)]:
        assert N.rmsnorm_train_bwd_workspace_bytes(T, 1, H, det) <= 16 << 20
    assert "16 MiB" in N.status_str(6)
