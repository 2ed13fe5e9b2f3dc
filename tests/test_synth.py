"""The seeded input generator: same seed -> same bytes, the views' strides, the recipes'
distributions (N(0,1) activations, 1 + 0.1*N(0,1) weights, 1 % of rows x16)."""
import numpy as np

import oracle
from rmsnorm_fwd_02_gb300 import synth


def test_same_seed_same_bytes_other_seed_differs():
    a = synth.make_case(3, 17, 64, residual=True, dh=True)
    b = synth.make_case(3, 17, 64, residual=True, dh=True)
    c = synth.make_case(4, 17, 64, residual=True, dh=True)
    for k in ("x", "dy", "w", "residual", "dh"):
        assert np.array_equal(getattr(a, k), getattr(b, k))
    assert not np.array_equal(a.x, c.x)


def test_dtypes_and_views():
    c = synth.tiny()
    assert c.x.dtype == np.uint16 and c.dy.dtype == np.uint16 and c.w.dtype == np.float32
    assert (c.T, c.nh, c.H, c.s_tok, c.s_head) == (64, 1, 256, 256, 256)
    p = synth.plain(65)
    assert p.w.dtype == np.uint16 and p.x.size == 65 * 4096
    s = synth.heads_strided(4)
    assert (s.nh, s.H, s.s_tok, s.s_head) == (24, 256, 8192, 256)
    assert s.x.size == 4 * 8192 and s.dy.size == 4 * 24 * 256
    h = synth.heads_contig(4)
    assert (h.nh, h.s_tok, h.s_head) == (4, 1024, 256)


def test_distributions():
    c = synth.make_case(0, 256, 1024, w_fp32=True)
    x = oracle.bf16_to_f64(c.x)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs(c.w.mean() - 1.0) < 0.02 and abs(c.w.std() - 0.1) < 0.02


def test_outlier_rows_scaled():
    c = synth.make_case(1, 400, 64, outlier_frac=0.01)
    x = oracle.bf16_to_f64(c.x).reshape(400, 64)
    rms = np.sqrt((x * x).mean(axis=1))
    assert int((rms > 6).sum()) == 4      # 1 % of 400 rows, scaled x16
