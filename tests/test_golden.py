"""The oracle reproduces tests/golden/oracle_small.txt bit for bit.

The fixture was written by tests/golden/make_golden.py, which calls only the oracle on
typed-in inputs.  It catches drift of the oracle between machines (the GPU host is
aarch64) and any later edit of its arithmetic.
"""
import os

import numpy as np

from golden import make_golden


def _read():
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small.txt")
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
