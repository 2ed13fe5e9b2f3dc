"""Writes tests/golden/layernorm_small.txt from the FP64 LayerNorm oracle alone.

The inputs are typed in below (small BF16-exact values, no random generator), so the
fixture pins the oracle's outputs bit for bit across machines (x86_64 here, aarch64 on
the GPU host) and across later edits of the oracle: any change to its arithmetic shows up
as a diff of this file and must be justified by the LayerNorm definition (textbook
LayerNorm with weight and bias; the op benchmarked beside RMSNorm in ROCm
TransformerEngine PR #478's normalization tables).

Run from the repository root:  python tests/golden/make_golden_layernorm.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402
from oracle import layernorm as OL  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "layernorm_small.txt")

R, H = 3, 8
EPS = float(np.float32(1e-5))
X = [[0.5, -1.25, 2.0, 0.0, 3.0, -0.75, 1.5, -2.5],
     [4.0, 4.0, 4.0, 4.0, 4.0, 4.0, 4.0, 4.0],
     [100.0, 101.0, 99.0, 100.5, 99.5, 100.0, 102.0, 98.0]]
DY = [[1.0, -0.5, 0.25, 2.0, -1.0, 0.75, 0.0, 1.5],
      [0.5, 0.5, -0.5, -0.5, 1.0, 1.0, -1.0, -1.0],
      [-2.0, 1.0, 0.125, 0.0, 3.0, -0.25, 0.5, -1.5]]
W = [1.0, 0.875, 1.125, 1.25, 0.75, 1.0, 0.9375, 1.0625]
B = [0.0, 0.125, -0.25, 0.5, -0.0625, 0.0, 1.0, -1.0]


def compute():
    x = oracle.round_bf16(np.array(X, np.float64).reshape(-1))
    dy = oracle.round_bf16(np.array(DY, np.float64).reshape(-1))
    w = np.array(W, np.float32)
    b = np.array(B, np.float32)
    out = {}
    y, mean, rstd = OL.fwd(x, w, b, EPS, R, H)
    out["fwd.mean"] = mean
    out["fwd.rstd"] = rstd
    out["fwd.y"] = y.reshape(-1)
    out["bwd.dx"] = OL.bwd_dx(x, dy, mean, rstd, w, R, H).reshape(-1)
    dw, db = OL.bwd_dw_db(x, dy, mean, rstd, R, H)
    out["bwd.dw"] = dw
    out["bwd.db"] = db
    return out


def main():
    out = compute()
    with open(OUT, "w") as f:
        f.write("# FP64 LayerNorm oracle outputs for the typed-in inputs of "
                "make_golden_layernorm.py.\n")
        f.write("# One line per tensor: name, then float.hex of each element.\n")
        for k, v in out.items():
            f.write(k + " " + " ".join(float(e).hex() for e in v) + "\n")
    print("wrote", OUT)


if __name__ == "__main__":
    main()
