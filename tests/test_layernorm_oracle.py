"""Pins of the FP64 LayerNorm oracle (oracle/layernorm_oracle.c) against what the
definition fixes independently of it: closed forms, finite differences, exact identities
and special cases -- and planted-mistake mutants of its source that the pins must reject.

LayerNorm (weight w, bias b) is the normalization beside RMSNorm in the ROCm
TransformerEngine PR #478 microbenchmark tables; the pages print no formula, so the pins
follow the textbook definition the oracle's header states.
"""
import numpy as np
import pytest

from oracle import layernorm as L
from oracle.build import LN_SRC, compile_c


def _rows(rng, R, H, scale=1.0, shift=0.0):
    return rng.standard_normal((R, H)) * scale + shift


# ---- closed forms ----------------------------------------------------------------------

def test_constant_row_gives_the_bias():
    # x_j = c: mean c, variance 0, rstd = 1/sqrt(eps) (eps = 1/4 -> exactly 2), y = b
    H = 8
    x = np.full((1, H), 0.375)
    w = np.linspace(0.5, 2.0, H)
    b = np.linspace(-1.0, 1.0, H)
    y, mean, rstd = L.fwd(x, w, b, 0.25, 1, H)
    assert mean[0] == 0.375 and rstd[0] == 2.0
    assert np.array_equal(y[0], b)


def test_two_valued_row_has_an_exact_rstd_and_output():
    # x = m + (a, -a, a, -a, ...): mean m, variance a^2; a = 3, eps = 7 -> rstd = 1/4;
    # y_j = +-(3/4) w_j + b_j.  m = 2^30 also pins the two-pass variance: the one-pass
    # E[x^2] - mean^2 loses the 9 entirely in FP64 (2^60 + 9 rounds to 2^60).
    H = 8
    w = np.array([1.0, 0.5, 2.0, 1.25, 0.75, 1.5, 0.25, 1.0])
    b = np.array([0.0, 1.0, -1.0, 0.5, -0.5, 2.0, 0.125, -2.0])
    sign = np.array([1.0, -1.0] * (H // 2))
    for m in (0.0, 2.0**30):
        x = (m + 3.0 * sign).reshape(1, H)
        y, mean, rstd = L.fwd(x, w, b, 7.0, 1, H)
        assert mean[0] == m and rstd[0] == 0.25, (m, mean[0], rstd[0])
        assert np.array_equal(y[0], 0.75 * sign * w + b)


# ---- gradients -------------------------------------------------------------------------

def _loss(x, w, b, dy, eps):
    R, H = x.shape
    y, _, _ = L.fwd(x, w, b, eps, R, H)
    return float((dy * y).sum())


@pytest.mark.parametrize("shape,eps", [((2, 8), 1e-5), ((3, 5), 0.3)])
def test_finite_difference_gradients(shape, eps):
    # central differences of L = sum(dy * y) match dx, dw and db
    rng = np.random.default_rng(3)
    R, H = shape
    x = _rows(rng, R, H, shift=0.5)
    w = 1.0 + 0.2 * rng.standard_normal(H)
    b = 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((R, H))
    _, mean, rstd = L.fwd(x, w, b, eps, R, H, want_y=False)
    dx = L.bwd_dx(x, dy, mean, rstd, w, R, H)
    dw, db = L.bwd_dw_db(x, dy, mean, rstd, R, H)
    h = 1e-6

    def fd(arr, idx):
        a = arr.copy(); a[idx] += h
        up = (a, w, b) if arr is x else ((x, a, b) if arr is w else (x, w, a))
        a2 = arr.copy(); a2[idx] -= h
        dn = (a2, w, b) if arr is x else ((x, a2, b) if arr is w else (x, w, a2))
        return (_loss(*up, dy, eps) - _loss(*dn, dy, eps)) / (2 * h)

    for i in range(R):
        for j in range(H):
            assert abs(fd(x, (i, j)) - dx[i, j]) <= 1e-6 * (1 + abs(dx[i, j]))
    for j in range(H):
        assert abs(fd(w, j) - dw[j]) <= 1e-6 * (1 + abs(dw[j]))
        assert abs(fd(b, j) - db[j]) <= 1e-6 * (1 + abs(db[j]))


def test_dx_identities():
    # sum_j dx_j = 0, and sum_j dx_j * xhat_j = H * c * eps * rstd^3 with c = mean(g * xhat)
    rng = np.random.default_rng(5)
    R, H, eps = 4, 64, 0.01
    x = _rows(rng, R, H, scale=0.2, shift=1.5)
    w = 1.0 + 0.1 * rng.standard_normal(H)
    b = np.zeros(H)
    dy = rng.standard_normal((R, H))
    _, mean, rstd = L.fwd(x, w, b, eps, R, H, want_y=False)
    dx = L.bwd_dx(x, dy, mean, rstd, w, R, H)
    xhat = (x - mean[:, None]) * rstd[:, None]
    c = (dy * w * xhat).mean(axis=1)
    scale = np.abs(dx).sum(axis=1)
    assert np.all(np.abs(dx.sum(axis=1)) <= 1e-12 * scale)
    want = H * c * eps * rstd**3
    assert np.allclose((dx * xhat).sum(axis=1), want, rtol=1e-9, atol=1e-12 * scale.max())


def test_single_row_and_zero_gradient():
    rng = np.random.default_rng(7)
    H = 16
    x = _rows(rng, 1, H)
    w = 1.0 + 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((1, H))
    _, mean, rstd = L.fwd(x, w, np.zeros(H), 1e-5, 1, H, want_y=False)
    dw, db = L.bwd_dw_db(x, dy, mean, rstd, 1, H)
    xhat = (x[0] - mean[0]) * rstd[0]
    assert np.array_equal(db, dy[0])
    assert np.allclose(dw, dy[0] * xhat, rtol=1e-15, atol=0)
    z = np.zeros((1, H))
    assert not L.bwd_dx(x, z, mean, rstd, w, 1, H).any()
    dw0, db0 = L.bwd_dw_db(x, z, mean, rstd, 1, H)
    assert not dw0.any() and not db0.any()


def test_bf16_and_fp32_inputs_read_exactly():
    # the same values as BF16 bits, FP32 and FP64 give the same results
    rng = np.random.default_rng(9)
    R, H = 3, 24
    xf = rng.standard_normal((R, H)).astype(np.float32)
    bits = (xf.view(np.uint32) >> 16).astype(np.uint16)          # truncate to BF16
    xb = (bits.astype(np.uint32) << 16).view(np.float32)
    w = np.linspace(0.5, 1.5, H).astype(np.float32)
    b = np.zeros(H, np.float32)
    r1 = L.fwd(bits, w, b, 1e-5, R, H)
    r2 = L.fwd(xb, w, b, 1e-5, R, H)
    r3 = L.fwd(xb.astype(np.float64), w.astype(np.float64), b.astype(np.float64), 1e-5, R, H)
    for a, c in zip(r1, r2):
        assert np.array_equal(a, c)
    for a, c in zip(r2, r3):
        assert np.array_equal(a, c)


PINS = [
    test_constant_row_gives_the_bias,
    test_two_valued_row_has_an_exact_rstd_and_output,
    lambda: test_finite_difference_gradients((2, 8), 1e-5),
    lambda: test_finite_difference_gradients((3, 5), 0.3),
    test_dx_identities,
    test_single_row_and_zero_gradient,
    test_bf16_and_fp32_inputs_read_exactly,
]

# (name, [(original text, mutated text), ...])
MUTANTS = [
    ("variance divisor H-1", [("const double var = ss / (double)H;",
                               "const double var = ss / (double)(H - 1);")]),
    ("one-pass variance", [("const double d = ln_ld(x, x_kind, r * H + j) - mu;\n      ss += d * d;",
                            "const double d = ln_ld(x, x_kind, r * H + j);\n      ss += d * d;"),
                           ("const double var = ss / (double)H;",
                            "const double var = ss / (double)H - mu * mu;")]),
    ("eps outside sqrt", [("1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)")]),
    ("no bias", [("ln_ld(b, b_kind, j);", "0.0;")]),
    ("y without the mean", [("y[r * H + j] = (ln_ld(x, x_kind, r * H + j) - mu) * rs",
                             "y[r * H + j] = ln_ld(x, x_kind, r * H + j) * rs")]),
    ("dx drops mean(g)", [("rs * (g[j] - gbar - xhat[j] * c)", "rs * (g[j] - xhat[j] * c)")]),
    ("dx drops xhat*c", [("rs * (g[j] - gbar - xhat[j] * c)", "rs * (g[j] - gbar)")]),
    ("dx sign", [("rs * (g[j] - gbar - xhat[j] * c)", "rs * (g[j] - gbar + xhat[j] * c)")]),
    ("g without w", [("g[j] = ln_ld(dy, dy_kind, r * H + j) * ln_ld(w, w_kind, j);",
                      "g[j] = ln_ld(dy, dy_kind, r * H + j);")]),
    ("c not a mean", [("const double c = gx / (double)H;", "const double c = gx;")]),
    ("dw without the mean", [("dw[j] += d * ((ln_ld(x, x_kind, r * H + j) - mu) * rs);",
                              "dw[j] += d * (ln_ld(x, x_kind, r * H + j) * rs);")]),
    ("db sums x", [("db[j] += d;", "db[j] += ln_ld(x, x_kind, r * H + j);")]),
]


def _build_mutant(tmp_path, edits):
    src = open(LN_SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor not unique/present: {old[:50]!r}"
        src = src.replace(old, new)
    path = tmp_path / "mut.c"
    path.write_text(src)
    return compile_c(str(path), str(tmp_path / "libmut.so"))


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, edits):
    L.use_library(_build_mutant(tmp_path, edits))
    failures = 0
    try:
        for pin in PINS:
            try:
                with np.errstate(all="ignore"):
                    pin()
            except AssertionError:
                failures += 1
    finally:
        L.use_library(None)
    assert failures > 0, f"no pin caught the planted mistake {name!r}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    L.use_library(_build_mutant(tmp_path, []))
    try:
        for pin in PINS:
            pin()
    finally:
        L.use_library(None)
