"""Pins the FP64 oracle to facts that do not come from the oracle itself.

The RMSNorm-training pages print no worked example, so the oracle is pinned by:
closed forms of the forward (zero row, constant row, a Pythagorean row), a central
finite-difference check of dx and dw against the forward, the exact identity
sum_j x_j*dx_j = rstd^3 * eps * sum_j x_j*g_j (which follows from the dx formula),
special cases (T = 1, dy = 0, constant rows), hand-made BF16 rounding ties, torch's
FP32 -> BF16 conversion on FP32-exact values, and per-head views against a reshaped
plain copy.  Each test names the plausible mistake it would catch.
"""
import math

import numpy as np
import pytest
import torch

import oracle

EPS = float(np.float32(1e-6))  # the op's eps is the FP32 value 1e-6


def bits(v):
    return int(oracle.round_bf16(np.array([v], np.float64))[0])


# ---- BF16 rounding ---------------------------------------------------------------------

def test_bf16_round_ties_and_single_rounding():
    # ties go to the even neighbour
    assert bits(1.0 + 2.0**-8) == 0x3F80            # between 1 and 1+2^-7 -> 1
    assert bits(1.0 + 3 * 2.0**-8) == 0x3F82        # between 1+2^-7 and 1+2^-6 -> 1+2^-6
    assert bits(-(1.0 + 3 * 2.0**-8)) == 0xBF82
    # just above a tie rounds up; an FP32 detour would land on the tie and go down
    assert bits(1.0 + 2.0**-8 + 2.0**-30) == 0x3F81
    assert bits(1.0 + 2.0**-8 - 2.0**-30) == 0x3F80
    # signed zero, overflow to inf, the largest finite value, subnormals
    assert bits(0.0) == 0x0000 and bits(-0.0) == 0x8000
    assert bits((2.0 - 2.0**-8) * 2.0**127) == 0x7F80
    assert bits((2.0 - 2.0**-8 - 2.0**-20) * 2.0**127) == 0x7F7F
    assert bits(2.0**-133) == 0x0001
    assert bits(2.0**-134) == 0x0000                 # tie between 0 and 2^-133 -> 0
    assert bits(3 * 2.0**-134) == 0x0002             # tie between 1 and 2 quanta -> 2
    assert bits(float("inf")) == 0x7F80
    assert bits(1.5) == 0x3FC0 and bits(-2.0) == 0xC000


def test_bf16_round_matches_torch_on_fp32_values():
    # torch rounds FP32 -> BF16 to nearest-even; on FP32-exact inputs one rounding from
    # FP64 must agree with it bit for bit.
    rng = np.random.default_rng(123)
    f = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e30).astype(np.float32),
        (rng.standard_normal(20000) * 1e-36).astype(np.float32),
    ])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(f.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_widening():
    b = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000], np.uint16)
    v = oracle.bf16_to_f64(b)
    assert v[0] == 1.0 and v[1] == -2.0 and v[2] == 2.0**-133
    assert v[3] == (2.0 - 2.0**-7) * 2.0**127 and math.copysign(1, v[4]) < 0


# ---- forward closed forms --------------------------------------------------------------

def _fwd64(x, w, eps=EPS, nh=1, s_tok=None, s_head=None, **kw):
    x = np.asarray(x, np.float64)
    T, H = x.shape[0], x.shape[-1]
    if s_tok is None:
        s_tok, s_head = H, H
    return oracle.fwd(x.reshape(-1), np.asarray(w, np.float64), eps, T, nh, H, s_tok,
                      s_head, **kw)


def test_fwd_zero_row():
    # zero row: rstd = 1/sqrt(eps), y = 0  (catches eps outside the sqrt)
    y, r, _ = _fwd64(np.zeros((1, 16)), np.ones(16))
    assert r[0] == 1.0 / math.sqrt(EPS)
    assert np.all(y == 0.0)


def test_fwd_constant_row():
    # constant row c: mean(x^2) = c^2, so rstd = 1/sqrt(c^2 + eps) and y_j = c*rstd*w_j
    # (catches a divisor of H-1 or a missing mean)
    H = 24
    w = np.linspace(0.5, 1.5, H)
    for c in (0.25, -3.0, 7.5):
        y, r, _ = _fwd64(np.full((1, H), c), w)
        rr = 1.0 / math.sqrt(c * c + EPS)
        assert r[0] == pytest.approx(rr, rel=1e-15)
        assert np.allclose(y[0], c * rr * w, rtol=1e-15, atol=0)


def test_fwd_pythagorean_row():
    # x = [3, 4, 0, 0]: sum of squares 25, mean 6.25
    # (eps chosen so that mean + eps is a perfect square: catches eps added outside the
    # mean or a sum of |x| instead of x^2)
    w = np.array([1.0, 2.0, 0.5, 1.0])
    y, r, _ = _fwd64(np.array([[3.0, 4.0, 0.0, 0.0]]), w, eps=-2.25)
    assert r[0] == 0.5                       # 1/sqrt(6.25 - 2.25) = 1/2
    assert np.array_equal(y[0], np.array([1.5, 4.0, 0.0, 0.0]))
    y, r, _ = _fwd64(np.array([[3.0, 4.0, 0.0, 0.0]]), w, eps=9.75)
    assert r[0] == 0.25                      # 1/sqrt(6.25 + 9.75) = 1/4


def test_fwd_row_subset_matches_full():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 40))
    w = rng.standard_normal(40)
    y, r, _ = _fwd64(x, w)
    rows = np.array([8, 0, 3])
    ys, rs, _ = _fwd64(x, w, rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(rs, r[rows])


def test_fwd_residual_sum_is_rounded_once_and_normalized():
    # h_new = BF16(x_in + res); the sum of two BF16 values is exact in FP64, so h is the
    # one rounding of the exact sum; the norm is then taken of h.
    H = 8
    xin = np.array([1.0, 1.0, 1.0, -1.5, 0.0, 2.0, 1.0, 0.5])
    res = np.array([2.0**-8, 3 * 2.0**-8, 1.0, 1.5, 0.0, -0.5, 2.0**-7, 0.25])
    xin_b = oracle.round_bf16(xin)
    res_b = oracle.round_bf16(res)
    w = np.ones(H, np.float32)
    y, r, h = oracle.fwd(xin_b, w, EPS, 1, 1, H, H, H, residual=res_b)
    want_h = np.array([0x3F80, 0x3F82, 0x4000, 0x0000, 0x0000, 0x3FC0, 0x3F81, 0x3F40],
                      np.uint16)
    assert np.array_equal(h[0], want_h)
    # the residual forward equals the plain forward on h
    y2, r2, _ = oracle.fwd(h[0], w, EPS, 1, 1, H, H, H)
    assert np.array_equal(y, y2) and np.array_equal(r, r2)


# ---- backward ----------------------------------------------------------------------

def _loss_fd_grads(x, w, dy, eps, dh=None, step=1e-6):
    """Central differences of L = sum(dy * y(x, w)) [+ sum(dh * x)] in FP64."""
    T, H = x.shape

    def L(xx, ww):
        y, _, _ = oracle.fwd(xx.reshape(-1), ww, eps, T, 1, H, H, H)
        v = float(np.sum(dy * y))
        if dh is not None:
            v += float(np.sum(dh * xx))
        return v

    gx = np.zeros_like(x)
    for t in range(T):
        for j in range(H):
            hs = step * max(1.0, abs(x[t, j]))
            xp, xm = x.copy(), x.copy()
            xp[t, j] += hs
            xm[t, j] -= hs
            gx[t, j] = (L(xp, w) - L(xm, w)) / (2 * hs)
    gw = np.zeros_like(w)
    for j in range(H):
        hs = step * max(1.0, abs(w[j]))
        wp, wm = w.copy(), w.copy()
        wp[j] += hs
        wm[j] -= hs
        gw[j] = (L(x, wp) - L(x, wm)) / (2 * hs)
    return gx, gw


@pytest.mark.parametrize("eps", [EPS, 0.3])
@pytest.mark.parametrize("shape", [(1, 4), (3, 16), (2, 7)])
def test_bwd_finite_difference(shape, eps):
    # Catches a wrong sign, a dropped term (x_hat * c), a wrong mean divisor, a missing
    # rstd factor, a transposed dy/x, and a dw that does not sum over rows.
    rng = np.random.default_rng(hash(shape) % 1000)
    T, H = shape
    x = rng.standard_normal((T, H))
    w = 1.0 + 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((T, H))
    _, r, _ = oracle.fwd(x.reshape(-1), w, eps, T, 1, H, H, H)
    dx = oracle.bwd_dx(x.reshape(-1), dy.reshape(-1), r, w, T, 1, H, H, H)
    dw = oracle.bwd_dw(x.reshape(-1), dy.reshape(-1), r, T, 1, H, H, H)
    gx, gw = _loss_fd_grads(x, w, dy, eps)
    scale_x = np.max(np.abs(gx))
    scale_w = np.max(np.abs(gw))
    assert np.max(np.abs(dx - gx)) <= 1e-7 * scale_x
    assert np.max(np.abs(dw - gw)) <= 1e-7 * scale_w


def test_bwd_residual_combined_gradient_fd():
    # residual form: the backward's input gradient is d/dh of sum(dy*y(h)) + sum(dh*h)
    rng = np.random.default_rng(11)
    T, H = 2, 12
    hx = rng.standard_normal((T, H))
    w = 1.0 + 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((T, H))
    dh = rng.standard_normal((T, H))
    _, r, _ = oracle.fwd(hx.reshape(-1), w, EPS, T, 1, H, H, H)
    dx = oracle.bwd_dx(hx.reshape(-1), dy.reshape(-1), r, w, T, 1, H, H, H,
                       dh=dh.reshape(-1))
    gx, _ = _loss_fd_grads(hx, w, dy, EPS, dh=dh)
    assert np.max(np.abs(dx - gx)) <= 1e-7 * np.max(np.abs(gx))


@pytest.mark.parametrize("eps", [EPS, 0.1, 2.0])
def test_bwd_identity_x_dot_dx(eps):
    # sum_j x_j*dx_j = rstd^3 * eps * sum_j x_j*g_j, g = dy*w (exact consequence of the
    # dx formula; vanishes as eps -> 0).  Catches c taken with the wrong normalization.
    rng = np.random.default_rng(7)
    T, H = 5, 64
    x = rng.standard_normal((T, H))
    w = 1.0 + 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((T, H))
    _, r, _ = oracle.fwd(x.reshape(-1), w, eps, T, 1, H, H, H)
    dx = oracle.bwd_dx(x.reshape(-1), dy.reshape(-1), r, w, T, 1, H, H, H)
    for t in range(T):
        lhs = float(np.dot(x[t], dx[t]))
        rhs = r[t] ** 3 * eps * float(np.dot(x[t], dy[t] * w))
        mag = float(np.dot(np.abs(x[t]), np.abs(dx[t]))) + abs(rhs)
        assert abs(lhs - rhs) <= 1e-12 * mag


def test_bwd_zero_upstream_gradient():
    rng = np.random.default_rng(3)
    T, H = 4, 32
    x = rng.standard_normal(T * H)
    w = rng.standard_normal(H)
    dy = np.zeros(T * H)
    r = np.full(T, 0.7)
    assert np.all(oracle.bwd_dx(x, dy, r, w, T, 1, H, H, H) == 0.0)
    assert np.all(oracle.bwd_dw(x, dy, r, T, 1, H, H, H) == 0.0)


def test_bwd_dw_single_row_and_constant_rows():
    # T = 1: dw_j = dy_j * x_j * rstd (catches summing the wrong axis)
    rng = np.random.default_rng(9)
    H = 16
    x = rng.standard_normal(H)
    dy = rng.standard_normal(H)
    r = np.array([0.37])
    dw = oracle.bwd_dw(x, dy, r, 1, 1, H, H, H)
    assert np.allclose(dw, dy * x * 0.37, rtol=1e-15, atol=0)
    # constant rows c_t with dy = 1 and rstd from the forward: dw_j = sum_t c_t/sqrt(c_t^2+eps)
    c = np.array([0.5, -2.0, 3.0, 0.125])
    T = c.size
    xc = np.repeat(c, H)
    _, rr, _ = oracle.fwd(xc, np.ones(H), EPS, T, 1, H, H, H)
    dw = oracle.bwd_dw(xc, np.ones(T * H), rr, T, 1, H, H, H)
    want = sum(ci / math.sqrt(ci * ci + EPS) for ci in c)
    assert np.allclose(dw, want, rtol=1e-14, atol=0)


def test_bwd_dh_is_added():
    rng = np.random.default_rng(4)
    T, H = 3, 8
    x, dy, dh = (rng.standard_normal(T * H) for _ in range(3))
    w = rng.standard_normal(H)
    r = np.array([1.1, 0.9, 0.5])
    a = oracle.bwd_dx(x, dy, r, w, T, 1, H, H, H)
    b = oracle.bwd_dx(x, dy, r, w, T, 1, H, H, H, dh=dh)
    assert np.allclose(b - a, dh.reshape(T, H), rtol=0, atol=1e-14)


# ---- per-head views ------------------------------------------------------------------

def test_per_head_strided_view_matches_reshaped_plain():
    # A [T, nh, Hd] view taking the first nh heads of a [T, bh*Hd] buffer must give what
    # the plain path gives on the gathered contiguous [T*nh, Hd] copy, bit for bit
    # (catches swapped strides and an off-by-one head index).
    rng = np.random.default_rng(21)
    T, bh, nh, Hd = 3, 5, 3, 16
    buf = oracle.round_bf16(rng.standard_normal(T * bh * Hd))
    dy = oracle.round_bf16(rng.standard_normal(T * nh * Hd))
    w = (1 + 0.1 * rng.standard_normal(Hd)).astype(np.float32)
    y, r, _ = oracle.fwd(buf, w, EPS, T, nh, Hd, bh * Hd, Hd)
    contig = buf.reshape(T, bh, Hd)[:, :nh, :].reshape(-1).copy()
    y2, r2, _ = oracle.fwd(contig, w, EPS, T * nh, 1, Hd, Hd, Hd)
    assert np.array_equal(y, y2) and np.array_equal(r, r2)
    dx = oracle.bwd_dx(buf, dy, r, w, T, nh, Hd, bh * Hd, Hd)
    dx2 = oracle.bwd_dx(contig, dy, r2, w, T * nh, 1, Hd, Hd, Hd)
    assert np.array_equal(dx, dx2)
    dw = oracle.bwd_dw(buf, dy, r, T, nh, Hd, bh * Hd, Hd)
    dw2 = oracle.bwd_dw(contig, dy, r2, T * nh, 1, Hd, Hd, Hd)
    assert np.array_equal(dw, dw2)
    # and the head-major stride (s_head != Hd) addresses the right element
    y3, _, _ = oracle.fwd(buf, w, EPS, T, nh, Hd, bh * Hd, Hd, rows=np.array([4]))
    t, h = divmod(4, nh)
    row = oracle.bf16_to_f64(buf.reshape(T, bh, Hd)[t, h])
    rr = 1.0 / math.sqrt(np.mean(row * row) + EPS)
    assert np.allclose(y3[0], row * rr * w.astype(np.float64), rtol=1e-15, atol=0)
