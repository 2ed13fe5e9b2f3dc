"""Helpers for the GPU parity tests: run the CUDA library through its C ABI on a seeded
case, run the FP64 oracle on the same bytes, and compare under the gates.

Gates (the op's stated accuracy, flashinfer PR #8827 description and Measurement; the
1-ulp and 1e-6 bounds are this build's tighter targets):
  y, dx   within 1 BF16 ulp of the FP64 result rounded to BF16 (ordinal distance <= 1);
          where g - xhat*c nearly cancels, dx may instead sit within the FP32 error of
          computing it, E_j = r*(2^-20*(|g_j| + |xhat_j*c|) + 2^-18*|xhat_j|*S) with
          S = mean_k |g_k*xhat_k| (the first term: the few roundings of g, xhat, the fma
          and the scaling; the second: the FP32 row reduction that forms c, whose error
          scales with the sum of |terms|), plus 2^-23*|dh_j| when dh is added and half a
          BF16 ulp for the final rounding
  rstd    |rstd - rstd64| <= 1e-6 * rstd64
  h       bit-exact (one rounding of an exact sum)
  dw      |dw - dw64| <= 1e-4 + 1e-4 * |dw64| for every element
The backward is fed rstd = FP32(rstd64), the oracle's own correctly rounded forward rstd,
so no oracle input ever comes from the CUDA path; the oracle's dx and dw use that same
FP32 value widened to FP64 (the gate).  dw against the oracle at rstd64 itself, the other
rstd form, is reported as dw_ratio_rstd64_*.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from rmsnorm_fwd_02_gb300 import _native as N

DEV = "cuda"
DW_ATOL = 1e-4
DW_RTOL = 1e-4
RSTD_RTOL = 1e-6


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(DEV).view(torch.bfloat16)


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return to_dev_bf16(a)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def wdtype(case) -> int:
    return N.RMSN_W_FP32 if case.w_fp32 else N.RMSN_W_BF16


def ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def sample_rows(R: int, n: int = 48, seed: int = 99) -> np.ndarray:
    if R <= 2 * n:
        return np.arange(R, dtype=np.int64)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(8, R - 8), size=n - 16, replace=False)
    return np.unique(np.concatenate([np.arange(8), np.arange(R - 8, R), mid])).astype(np.int64)


class DeviceCase:
    """The case's inputs resident on the GPU."""

    def __init__(self, case):
        self.c = case
        self.x = to_dev(case.x)
        self.dy = to_dev(case.dy)
        self.w = to_dev(case.w)
        self.res = None if case.residual is None else to_dev(case.residual)
        self.dh = None if case.dh is None else to_dev(case.dh)


def gpu_fwd(dc: DeviceCase, residual: bool):
    c = dc.c
    R, H = c.R, c.H
    y = torch.empty(R * H, dtype=torch.bfloat16, device=DEV)
    rstd = torch.empty(R, dtype=torch.float32, device=DEV)
    h = torch.empty(R * H, dtype=torch.bfloat16, device=DEV) if residual else None
    N.rmsnorm_train_fwd(dc.x, dc.res if residual else None, dc.w, wdtype(c), y, h, rstd,
                        c.T, c.nh, H, c.s_tok, c.s_head, c.eps)
    return y, rstd, h


def gpu_bwd(dc: DeviceCase, x_dev, s_tok, s_head, rstd_dev, deterministic, with_dh=False):
    c = dc.c
    R, H = c.R, c.H
    dx = torch.empty(R * H, dtype=torch.bfloat16, device=DEV)
    dw = torch.empty(H, dtype=torch.float32, device=DEV)
    nbytes = N.rmsnorm_train_bwd_workspace_bytes(c.T, c.nh, H, deterministic)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    N.rmsnorm_train_bwd(x_dev, dc.dy, dc.dh if with_dh else None, rstd_dev, dc.w, wdtype(c),
                        dx, dw, ws, nbytes, c.T, c.nh, H, s_tok, s_head, deterministic)
    return dx, dw


def check_rstd(rstd_gpu: np.ndarray, rstd64: np.ndarray):
    rel = np.abs(rstd_gpu.astype(np.float64) - rstd64) / rstd64
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= RSTD_RTOL, f"rstd rel err {worst:.3e} > {RSTD_RTOL}"
    return worst


def check_bf16_1ulp(gpu_bits: np.ndarray, ref64: np.ndarray, what: str, extra_ok=None):
    """Ordinal distance <= 1 from BF16_RNE(ref64); elements beyond it pass only if
    |gpu - ref64| <= extra_ok + half a BF16 ulp of the GPU value.  Returns the largest
    ordinal distance, the count that needed the second clause, and their worst ratio of
    error to allowance."""
    ref_bits = oracle.round_bf16(ref64)
    d = np.abs(ordinal(gpu_bits.reshape(-1)) - ordinal(ref_bits.reshape(-1)))
    bad = d > 1
    n_extra = 0
    worst = 0.0
    if extra_ok is not None and bad.any():
        gv = oracle.bf16_to_f64(gpu_bits.reshape(-1))
        err = np.abs(gv - ref64.reshape(-1))
        allow = extra_ok.reshape(-1) + np.abs(gv) * 2.0**-8
        ok2 = err <= allow
        n_extra = int((bad & ok2).sum())
        worst = float((err[bad] / allow[bad]).max())
        bad = bad & ~ok2
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} elements beyond 1 BF16 ulp and the FP32 cancellation "
        f"allowance (max ordinal distance {int(d.max())}, worst err/allowance {worst:.3f})")
    return int(d.max()) if d.size else 0, n_extra, worst


def dx_cancel_tol(x_bits, dy_bits, w, r, H, dh_bits=None):
    """E_j of the module docstring: the FP32 error of evaluating dx_j, per element."""
    xv = oracle.bf16_to_f64(x_bits).reshape(-1, H)
    dyv = oracle.bf16_to_f64(dy_bits).reshape(-1, H)
    wv = oracle.bf16_to_f64(w) if w.dtype == np.uint16 else w.astype(np.float64)
    rr = r.reshape(-1, 1)
    xh = xv * rr
    g = dyv * wv
    c = (g * xh).mean(axis=1, keepdims=True)
    S = np.abs(g * xh).mean(axis=1, keepdims=True)
    E = rr * (2.0**-20 * (np.abs(g) + np.abs(xh * c)) + 2.0**-18 * np.abs(xh) * S)
    if dh_bits is not None:
        E = E + 2.0**-23 * np.abs(oracle.bf16_to_f64(dh_bits).reshape(-1, H))
    return E


def check_dw(dw_gpu: np.ndarray, dw64: np.ndarray):
    err = np.abs(dw_gpu.astype(np.float64) - dw64)
    budget = DW_ATOL + DW_RTOL * np.abs(dw64)
    ratio = float((err / budget).max())
    assert ratio <= 1.0, f"dw worst err/budget {ratio:.4f} > 1"
    return ratio


def gather_rows(flat: np.ndarray, case, rows: np.ndarray) -> np.ndarray:
    """Rows of a strided activation buffer as a contiguous [len(rows), H] array."""
    t = rows // case.nh
    h = rows % case.nh
    base = t * case.s_tok + h * case.s_head
    idx = base[:, None] + np.arange(case.H)[None, :]
    return flat[idx]


def report(rec: dict):
    path = os.environ.get("RMSN_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def eager_fp32_dw(xs_dev, dy_dev, r_dev, c, s_tok, s_head):
    """dw the plain FP32 way (torch on the GPU: x*rstd, times dy, summed over rows by
    torch's reduction): the pages' FP32 eager reference, whose worst dw error a kernel's
    must not exceed."""
    R, H = c.R, c.H
    x = torch.as_strided(xs_dev, (c.T, c.nh, H), (s_tok, s_head, 1)).reshape(R, H).float()
    xhat = x * r_dev.view(R, 1)
    return (dy_dev.view(R, H).float() * xhat).sum(dim=0)


def run_case(case, modes=(True, False), full_rows_limit=4096 * 4096, with_dh=False,
             check_eager=False):
    """Forward + backward of `case` on the GPU against the oracle.  Rows beyond
    `full_rows_limit` elements are sampled for y / h / dx; rstd and dw are checked in
    full.  With check_eager, each mode's worst dw error must also be at most the FP32
    eager reference's.  Returns a dict of the worst figures."""
    c = case
    R, H = c.R, c.H
    residual = c.residual is not None
    dc = DeviceCase(c)
    full = R * H <= full_rows_limit
    rows = None if full else sample_rows(R)
    out = {"case": c.label, "T": c.T, "nh": c.nh, "H": H, "R": R}

    # ---- forward ----
    y, rstd, h = gpu_fwd(dc, residual)
    torch.cuda.synchronize()
    _, rstd64, h_all = oracle.fwd(c.x, c.w, c.eps, c.T, c.nh, H, c.s_tok, c.s_head,
                                  residual=c.residual, want_y=False)
    rstd_g = rstd.cpu().numpy()
    out["rstd_rel"] = check_rstd(rstd_g, rstd64)
    y64, _, h_bits = oracle.fwd(c.x, c.w, c.eps, c.T, c.nh, H, c.s_tok, c.s_head,
                                residual=c.residual, rows=rows)
    yb = bits_of(y).reshape(R, H)
    out["y_ulp"], _, _ = check_bf16_1ulp(yb if rows is None else yb[rows], y64, "y")
    if residual:
        hb = bits_of(h).reshape(R, H)
        assert np.array_equal(hb, h_all.reshape(R, H)), "h not bit-exact"

    # ---- backward: saved input is x (plain) or the oracle's h (residual) ----
    if residual:
        xs_bits = h_all.reshape(-1)
        xs_dev = to_dev(xs_bits)
        s_tok, s_head = c.nh * H, H
    else:
        xs_bits = c.x
        xs_dev = dc.x
        s_tok, s_head = c.s_tok, c.s_head
    r32 = rstd64.astype(np.float32)
    r_in = r32.astype(np.float64)
    r_dev = to_dev(r32)
    dw64 = oracle.bwd_dw(xs_bits, c.dy, r_in, c.T, c.nh, H, s_tok, s_head)
    # the second rstd form: the FP64 rstd itself (reported, not gated -- the kernels are
    # handed the FP32 rstd a forward returns)
    dw64_exact = oracle.bwd_dw(xs_bits, c.dy, rstd64, c.T, c.nh, H, s_tok, s_head)
    dx64 = oracle.bwd_dx(xs_bits, c.dy, r_in, c.w, c.T, c.nh, H, s_tok, s_head,
                         dh=c.dh if with_dh else None, rows=rows)
    sel = np.arange(R) if rows is None else rows
    xrows = gather_rows(xs_bits, c, sel) if not residual else xs_bits.reshape(R, H)[sel]
    tol = dx_cancel_tol(xrows, c.dy.reshape(R, H)[sel], c.w, r_in[sel], H,
                        dh_bits=c.dh.reshape(R, H)[sel] if with_dh else None)
    eager_err = None
    if check_eager:
        dw_e = eager_fp32_dw(xs_dev, dc.dy, r_dev, c, s_tok, s_head).cpu().numpy()
        eager_err = float(np.abs(dw_e.astype(np.float64) - dw64).max())
        out["dw_eager_fp32_max_err"] = eager_err
    dws = {}
    for det in modes:
        dx, dw = gpu_bwd(dc, xs_dev, s_tok, s_head, r_dev, det, with_dh=with_dh)
        torch.cuda.synchronize()
        dxb = bits_of(dx).reshape(R, H)
        ulp, n_extra, worst = check_bf16_1ulp(dxb[sel], dx64, f"dx (det={det})",
                                              extra_ok=tol)
        ratio = check_dw(dw.cpu().numpy(), dw64)
        dws[det] = (dxb, dw.cpu().numpy())
        key = "det" if det else "nondet"
        budget = DW_ATOL + DW_RTOL * np.abs(dw64_exact)
        out[f"dw_ratio_rstd64_{key}"] = float(
            (np.abs(dw.cpu().numpy().astype(np.float64) - dw64_exact) / budget).max())
        if eager_err is not None:
            err = float(np.abs(dw.cpu().numpy().astype(np.float64) - dw64).max())
            out[f"dw_max_err_{key}"] = err
            assert err <= eager_err, (
                f"dw worst error {err:.3e} above the FP32 eager reference's {eager_err:.3e}")
        out[f"dx_ulp_{key}"] = ulp
        out[f"dx_cancel_{key}"] = n_extra
        out[f"dx_cancel_worst_{key}"] = worst
        out[f"dw_ratio_{key}"] = ratio
    if len(dws) == 2:
        # the two modes share the row pass: dx is bit-identical
        assert np.array_equal(dws[True][0], dws[False][0]), "dx differs between modes"
    assert N.rmsnorm_train_device_error(reset=True) == 0
    report(out)
    return out
