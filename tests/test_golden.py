"""The oracles reproduce tests/golden/oracle_small.txt and layernorm_small.txt bit for bit.

The fixtures were written by tests/golden/make_golden.py and make_golden_layernorm.py,
which call only the oracle on typed-in inputs.  It catches drift of the oracle between machines (the GPU host is
aarch64) and any later edit of its arithmetic.
"""
import os

import numpy as np

from golden import make_golden, make_golden_layernorm


def _read(name="oracle_small.txt"):
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, *vals = line.split()
            out[name] = np.array([float.fromhex(v) for v in vals])
    return out


def test_oracle_matches_golden_bitwise():
    want = _read()
    got = make_golden.compute()
    assert set(want) == set(got)
    for k in want:
        assert np.array_equal(want[k], got[k]), k


def test_layernorm_oracle_matches_golden_bitwise():
    want = _read("layernorm_small.txt")
    got = make_golden_layernorm.compute()
    assert set(want) == set(got)
    for k in want:
        assert np.array_equal(want[k], got[k]), k
