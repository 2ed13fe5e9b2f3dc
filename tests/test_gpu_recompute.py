"""GPU parity of the backward that recomputes rstd (rmsnorm_train_bwd_recompute): the
checkpointed step of flashinfer PR #8827's Measurement section (forward, forward again,
backward) with the second forward folded into the backward.

Gates: its rstd within 1e-6 relative of the FP64 value (the forward's gate); dx and dw
within the gates of tests/parity.py against the oracle at FP32(rstd64), the rstd a
correctly rounded forward returns, on every element; dx bit-identical across modes; the
deterministic mode bit-identical over repeated runs."""
import numpy as np
import pytest
import torch

from rmsnorm_fwd_02_gb300 import _native as N
from rmsnorm_fwd_02_gb300 import synth
import parity

pytestmark = pytest.mark.gpu


CASES = {
    "tiny_T64_H256": (lambda: synth.tiny(), False),                  # one-launch small path
    "plain_T1_H4096": (lambda: synth.plain(1), False),
    "plain_T257_H4096": (lambda: synth.plain(257), False),
    "plain_T16384_H4096": (lambda: synth.plain(16384), False),
    "stress_T131072_H1536": (lambda: synth.stress(131072, 1536), False),
    "stress_T32768_H5120": (lambda: synth.stress(32768, 5120), False),
    "residual_T96_H6144_dh": (lambda: synth.residual(96, with_dh=True), True),
    "residual_T7168_H6144_dh": (lambda: synth.residual(7168, with_dh=True), True),
    "residual_T7168_H6144": (lambda: synth.residual(7168), False),
    "heads24of32_T4096": (lambda: synth.heads_strided(4096), False),
    "heads4_T4096": (lambda: synth.heads_contig(4096), False),
    "w8_T5003": (lambda: synth.make_case(13, 5003, 8, label="w8_T5003"), False),
    "w264_T4500": (lambda: synth.make_case(13, 4500, 264, label="w264_T4500"), False),
    "w8192_T300": (lambda: synth.make_case(17, 300, 8192, w_fp32=True, label="w8192"), False),
}


@pytest.mark.parametrize("name", list(CASES))
def test_recompute_parity(name):
    mk, with_dh = CASES[name]
    parity.run_case(mk(), with_dh=with_dh, recompute=True)


@pytest.mark.parametrize("mk", [lambda: synth.plain(4096), lambda: synth.tiny()])
def test_recompute_deterministic_bits(mk):
    c = mk()
    dc = parity.DeviceCase(c)
    ref = None
    for _ in range(10):
        dx, dw, rs = parity.gpu_bwd_recompute(dc, dc.x, c.s_tok, c.s_head, True)
        cur = (parity.bits_of(dx), dw.cpu().numpy().view(np.uint32),
               rs.cpu().numpy().view(np.uint32))
        if ref is None:
            ref = cur
        else:
            for a, b in zip(ref, cur):
                assert np.array_equal(a, b)
    dxn, _, rsn = parity.gpu_bwd_recompute(dc, dc.x, c.s_tok, c.s_head, False)
    assert np.array_equal(ref[0], parity.bits_of(dxn))
    assert np.array_equal(ref[2], rsn.cpu().numpy().view(np.uint32))
    assert N.rmsnorm_train_device_error(reset=True) == 0


def test_recompute_rejects_missing_rstd_out():
    c = synth.plain(300)
    dc = parity.DeviceCase(c)
    dx = torch.empty(c.R * c.H, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(c.H, dtype=torch.float32, device="cuda")
    with pytest.raises(N.RmsnError) as ei:
        N.rmsnorm_train_bwd_recompute(dc.x, dc.dy, None, dc.w, N.RMSN_W_BF16, dx, dw, None,
                                      None, 0, c.T, 1, c.H, c.H, c.H, 1e-6, True)
    assert ei.value.status == 1


def test_autograd_recompute_rstd_matches_direct_calls():
    import rmsnorm_fwd_02_gb300 as R
    c = synth.plain(300)
    dc = parity.DeviceCase(c)
    x = dc.x.view(c.T, c.H).clone().requires_grad_(True)
    w = dc.w.clone().requires_grad_(True)
    y = R.rmsnorm_train(x, w, c.eps, deterministic=True, recompute_rstd=True)
    dy = dc.dy.view(c.T, c.H)
    y.backward(dy)
    dx0, dw0, rs0 = R.rmsnorm_bwd_recompute(dy, dc.x.view(c.T, c.H), dc.w, c.eps, True)
    _, rstd = R.rmsnorm_fwd(dc.x.view(c.T, c.H), dc.w, c.eps)
    assert torch.equal(x.grad, dx0)
    assert torch.equal(w.grad, dw0.to(w.dtype))
    rel = ((rs0 - rstd).abs() / rstd).max().item()
    assert rel <= 2.0**-22, rel
