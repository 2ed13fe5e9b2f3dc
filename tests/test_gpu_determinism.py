"""Determinism and bitwise invariants of the CUDA path (no oracle needed).

- deterministic=True: dx and dw bit-identical over 10 runs (the op's det mode contract,
  flashinfer PR #8827 description; its test list checks det bit for bit twice).
- both modes run the same forward and the same row pass: dx identical across modes.
- per-head views equal the plain path on a gathered contiguous copy, bit for bit (y,
  rstd, dx; dw too in deterministic mode, where the partition depends on R and H only).
- the residual form's y and rstd equal the plain forward run on its h (to 2^-22 in rstd,
  1 BF16 ulp in y: the two forms may split a row over threads differently).
- a training step captured in a CUDA graph replays to the same bits as direct calls.
"""
import numpy as np
import pytest
import torch

from rmsnorm_fwd_02_gb300 import _native as N
from rmsnorm_fwd_02_gb300 import synth
import parity

pytestmark = pytest.mark.gpu


def _bits(t):
    return parity.bits_of(t)


DET_CASES = {
    "tiny_T64_H256": (lambda: synth.tiny(), False),                # one-launch small path
    "plain_T4096_H4096": (lambda: synth.plain(4096), False),
    "plain_T65536_H4096": (lambda: synth.plain(65536), False),     # the headline workload
    "stress_T32768_H5120": (lambda: synth.stress(32768, 5120), False),
    "residual_T7168_H6144": (lambda: synth.residual(7168, with_dh=True), False),
    "residual_T7168_H6144_dh": (lambda: synth.residual(7168, with_dh=True), True),
    "residual_T96_H6144_dh": (lambda: synth.residual(96, with_dh=True), True),
    "heads24of32_T4096": (lambda: synth.heads_strided(4096), False),
    "heads4_T4096": (lambda: synth.heads_contig(4096), False),
    "heads4_T65536": (lambda: synth.heads_contig(65536), False),
}


@pytest.mark.parametrize("name", list(DET_CASES))
def test_det_bitwise_10_runs(name):
    mk, with_dh = DET_CASES[name]
    c = mk()
    residual = c.residual is not None
    dc = parity.DeviceCase(c)
    y, rstd, h = parity.gpu_fwd(dc, residual)
    assert N.rmsnorm_train_device_error(reset=True) == 0   # (a wait that gave up, if any)
    # the backward's saved input: x itself, or h of the residual form
    xs, s_tok, s_head = (h, c.nh * c.H, c.H) if residual else (dc.x, c.s_tok, c.s_head)
    ref = None
    for _ in range(10):
        dx, dw = parity.gpu_bwd(dc, xs, s_tok, s_head, rstd, True, with_dh=with_dh)
        cur = (_bits(dx), dw.cpu().numpy().view(np.uint32))
        if ref is None:
            ref = cur
        else:
            assert np.array_equal(ref[0], cur[0]) and np.array_equal(ref[1], cur[1])
    assert N.rmsnorm_train_device_error(reset=True) == 0
    y2, rstd2, h2 = parity.gpu_fwd(dc, residual)
    assert N.rmsnorm_train_device_error(reset=True) == 0
    assert np.array_equal(_bits(y), _bits(y2))
    assert torch.equal(rstd, rstd2)
    if residual:
        assert np.array_equal(_bits(h), _bits(h2))
    # non-deterministic mode: same dx bits
    dxn, _ = parity.gpu_bwd(dc, xs, s_tok, s_head, rstd, False, with_dh=with_dh)
    assert np.array_equal(ref[0], _bits(dxn))
    assert N.rmsnorm_train_device_error(reset=True) == 0


@pytest.mark.parametrize("strided", [True, False])
def test_per_head_equals_plain_bitwise(strided):
    c = synth.heads_strided(1024) if strided else synth.heads_contig(1024)
    dc = parity.DeviceCase(c)
    y, rstd, _ = parity.gpu_fwd(dc, False)
    dx, dw = parity.gpu_bwd(dc, dc.x, c.s_tok, c.s_head, rstd, True)
    # gathered contiguous copy as plain rows [T*nh, 256]
    rows = np.arange(c.R)
    flat = parity.gather_rows(c.x, c.nh, c.H, c.s_tok, c.s_head, rows).reshape(-1)
    p = synth.Case(T=c.R, nh=1, H=c.H, s_tok=c.H, s_head=c.H, x=flat, dy=c.dy, w=c.w)
    dp = parity.DeviceCase(p)
    y2, rstd2, _ = parity.gpu_fwd(dp, False)
    dx2, dw2 = parity.gpu_bwd(dp, dp.x, p.s_tok, p.s_head, rstd2, True)
    assert np.array_equal(_bits(y), _bits(y2))
    assert torch.equal(rstd, rstd2)
    assert np.array_equal(_bits(dx), _bits(dx2))
    assert torch.equal(dw, dw2)


def test_residual_forward_equals_plain_on_h():
    c = synth.residual(300)
    dc = parity.DeviceCase(c)
    y, rstd, h = parity.gpu_fwd(dc, True)
    p = synth.Case(T=c.T, nh=1, H=c.H, s_tok=c.H, s_head=c.H, x=_bits(h), dy=c.dy, w=c.w)
    dp = parity.DeviceCase(p)
    y2, rstd2, _ = parity.gpu_fwd(dp, False)
    # the statistics come from h: the two forms may split a row over threads differently
    # (the residual form stages twice the bytes a row), so their FP32 sums of squares may
    # round differently -- rstd within 2^-22 relative, y within 1 BF16 ulp
    rel = ((rstd - rstd2).abs() / rstd2).max().item()
    assert rel <= 2.0**-22, rel
    d = np.abs(parity.ordinal(_bits(y)) - parity.ordinal(_bits(y2)))
    assert d.max() <= 1


def test_empty_input_zero_fills_dw():
    c = synth.make_case(0, 0, 512)
    dc = parity.DeviceCase(synth.make_case(0, 1, 512))
    dw = torch.full((512,), 7.0, device="cuda")
    dx = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(1, device="cuda")
    for det in (0, 1):
        N.rmsnorm_train_bwd(dc.x, dc.dy, None, rstd, dc.w, N.RMSN_W_BF16, dx, dw, None, 0,
                            0, 1, 512, 512, 512, det)
        torch.cuda.synchronize()
        assert torch.count_nonzero(dw).item() == 0
        dw.fill_(7.0)
    # forward with T = 0 is a no-op
    y = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    N.rmsnorm_train_fwd(dc.x, None, dc.w, N.RMSN_W_BF16, y, None, rstd, 0, 1, 512, 512, 512,
                        1e-6)
    assert c.R == 0


def test_workspace_too_small_is_rejected():
    c = synth.plain(300)      # above the one-launch (no workspace) size
    dc = parity.DeviceCase(c)
    need = N.rmsnorm_train_bwd_workspace_bytes(c.T, 1, c.H, True)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dx = torch.empty(c.R * c.H, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(c.H, dtype=torch.float32, device="cuda")
    rstd = torch.ones(c.R, device="cuda")
    # the query covers both launch shapes (with and without dh); here the dh shape needs
    # all of it, and any call needs more than 16 bytes
    for dh, nbytes in ((dc.dy, need - 16), (None, 16)):
        with pytest.raises(N.RmsnError) as ei:
            N.rmsnorm_train_bwd(dc.x, dc.dy, dh, rstd, dc.w, N.RMSN_W_BF16, dx, dw, ws,
                                nbytes, c.T, 1, c.H, c.H, c.H, True)
        assert ei.value.status == 3
    for dh in (dc.dy, None):   # the queried size is accepted either way
        N.rmsnorm_train_bwd(dc.x, dc.dy, dh, rstd, dc.w, N.RMSN_W_BF16, dx, dw, ws, need,
                            c.T, 1, c.H, c.H, c.H, True)
    torch.cuda.synchronize()
    assert N.rmsnorm_train_device_error(reset=True) == 0


def test_autograd_wrapper_matches_direct_calls():
    import rmsnorm_fwd_02_gb300 as R
    c = synth.plain(100)
    dc = parity.DeviceCase(c)
    x = dc.x.view(c.T, c.H).clone().requires_grad_(True)
    w = dc.w.clone().requires_grad_(True)
    y = R.rmsnorm_train(x, w, 1e-6, deterministic=True)
    dy = dc.dy.view(c.T, c.H)
    y.backward(dy)
    y0, rstd0 = R.rmsnorm_fwd(dc.x.view(c.T, c.H), dc.w)
    dx0, dw0 = R.rmsnorm_bwd(dy, dc.x.view(c.T, c.H), rstd0, dc.w, True)
    assert torch.equal(y, y0)
    assert torch.equal(x.grad, dx0)
    assert torch.equal(w.grad, dw0.to(w.dtype))


@pytest.mark.parametrize("det", [True, False])
def test_cuda_graph_replay_matches_direct_calls(det):
    # forward + backward enqueued on a side stream under stream capture (the launches use
    # programmatic dependent launch attributes) and replayed: the same bits as direct calls
    # (T=16384: 35 stages a CTA, so the non-deterministic backward opens its row pool, whose
    # per-call tag a replay repeats)
    c = synth.plain(16384)
    dc = parity.DeviceCase(c)
    R, H = c.R, c.H
    nbytes = N.rmsnorm_train_bwd_workspace_bytes(c.T, 1, H, det)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    y = torch.empty(R * H, dtype=torch.bfloat16, device="cuda")
    rstd = torch.empty(R, dtype=torch.float32, device="cuda")
    dx = torch.empty(R * H, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(H, dtype=torch.float32, device="cuda")

    def step(stream):
        N.rmsnorm_train_fwd(dc.x, None, dc.w, N.RMSN_W_BF16, y, None, rstd, c.T, 1, H, H, H,
                            c.eps, stream=stream)
        N.rmsnorm_train_bwd(dc.x, dc.dy, None, rstd, dc.w, N.RMSN_W_BF16, dx, dw, ws, nbytes,
                            c.T, 1, H, H, H, det, stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s.cuda_stream)   # warm-up: kernel attributes set outside the capture
    torch.cuda.synchronize()
    want = (_bits(y), rstd.cpu().numpy().copy(), _bits(dx), dw.cpu().numpy().copy())
    for t in (y, dx):
        t.zero_()
    rstd.zero_()
    dw.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s.cuda_stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    got = (_bits(y), rstd.cpu().numpy(), _bits(dx), dw.cpu().numpy())
    assert np.array_equal(want[0], got[0]) and np.array_equal(want[1], got[1])
    assert np.array_equal(want[2], got[2])
    if det:
        assert np.array_equal(want[3], got[3])
    else:
        # rows go to CTAs as they come, so the partials (and dw's last bits) vary from run
        # to run; each run sits within the dw budget of the FP64 sum
        np.testing.assert_allclose(got[3], want[3], rtol=parity.DW_RTOL, atol=parity.DW_ATOL)
    assert N.rmsnorm_train_device_error(reset=True) == 0


@pytest.mark.parametrize("mk", [lambda: synth.stress(4096, 1536), lambda: synth.plain(300),
                                lambda: synth.heads_strided(512),
                                lambda: synth.make_case(9, 2000, 8192, w_fp32=True),
                                lambda: synth.plain(16384)],   # the row pool opened
                         ids=["stress4096", "plain300", "heads512", "w32_H8192", "plain16384"])
def test_nondet_workspace_needs_no_initial_contents_and_is_reusable(mk):
    # the non-deterministic backward zeroes its own row counter on the stream: a workspace
    # full of garbage, and the same workspace reused by calls queued back to back, give dx
    # bit-equal to the deterministic mode's and dw within the budget of the same sum
    c = mk()
    dc = parity.DeviceCase(c)
    _, rstd, _ = parity.gpu_fwd(dc, False)
    dx_d, dw_d = parity.gpu_bwd(dc, dc.x, c.s_tok, c.s_head, rstd, True)
    nbytes = N.rmsnorm_train_bwd_workspace_bytes(c.T, c.nh, c.H, False)
    assert nbytes == 16 + N.rmsnorm_train_bwd_workspace_bytes(c.T, c.nh, c.H, True)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):   # queued back to back on one stream, one workspace
        dx = torch.empty_like(dx_d)
        dw = torch.empty_like(dw_d)
        N.rmsnorm_train_bwd(dc.x, dc.dy, None, rstd, dc.w, parity.wdtype(c), dx, dw, ws,
                            nbytes, c.T, c.nh, c.H, c.s_tok, c.s_head, False)
        outs.append((dx, dw))
    torch.cuda.synchronize()
    for dx, dw in outs:
        assert torch.equal(dx.view(torch.int16), dx_d.view(torch.int16))
        # both modes sit within the dw budget of the FP64 sum (the parity tests check
        # that); a sum that kept an earlier call's value or garbage would be far outside
        torch.testing.assert_close(dw, dw_d, rtol=parity.DW_RTOL, atol=parity.DW_ATOL)
    assert N.rmsnorm_train_device_error(reset=True) == 0


def test_nondet_workspace_too_small_is_rejected():
    c = synth.plain(300)
    dc = parity.DeviceCase(c)
    need = N.rmsnorm_train_bwd_workspace_bytes(c.T, 1, c.H, False)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dx = torch.empty(c.R * c.H, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(c.H, dtype=torch.float32, device="cuda")
    rstd = torch.ones(c.R, device="cuda")
    with pytest.raises(N.RmsnError) as ei:
        # the counter alone, without room for the partials
        N.rmsnorm_train_bwd(dc.x, dc.dy, None, rstd, dc.w, N.RMSN_W_BF16, dx, dw, ws, 16,
                            c.T, 1, c.H, c.H, c.H, False)
    assert ei.value.status == 3
    N.rmsnorm_train_bwd(dc.x, dc.dy, None, rstd, dc.w, N.RMSN_W_BF16, dx, dw, ws, need,
                        c.T, 1, c.H, c.H, c.H, False)
    torch.cuda.synchronize()
    assert N.rmsnorm_train_device_error(reset=True) == 0
