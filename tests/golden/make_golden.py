"""Writes tests/golden/oracle_small.txt from the FP64 oracle alone.

The inputs are typed in below (small BF16-exact values, no random generator), so the
fixture pins the oracle's outputs bit for bit across machines (x86_64 here, aarch64 on
the GPU host) and across later edits of the oracle: any change to its arithmetic shows
up as a diff of this file and must be justified by the op's definition (flashinfer PR
#8827, description: forward y and rstd, fused residual h_new, backward dx and dw).

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.txt")

T, H = 3, 8
EPS = float(np.float32(1e-6))
X = [[0.5, -1.25, 2.0, 0.0, 3.0, -0.75, 1.5, -2.5],
     [0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0],
     [1.0, 1.0, 1.0, 1.0, -1.0, -1.0, -1.0, -1.0]]
RES = [[0.25, 0.25, -1.0, 0.125, 2.0, 0.75, -0.5, 0.5],
       [1.0, -2.0, 0.5, 0.0, 4.0, 0.0, 0.0, -0.25],
       [0.00390625, 0.01171875, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0]]
DY = [[1.0, -0.5, 0.25, 2.0, -1.0, 0.75, 0.0, 1.5],
      [0.5, 0.5, -0.5, -0.5, 1.0, 1.0, -1.0, -1.0],
      [-2.0, 1.0, 0.125, 0.0, 3.0, -0.25, 0.5, -1.5]]
W = [1.0, 0.875, 1.125, 1.25, 0.75, 1.0, 0.9375, 1.0625]


def compute():
    x = oracle.round_bf16(np.array(X, np.float64).reshape(-1))
    res = oracle.round_bf16(np.array(RES, np.float64).reshape(-1))
    dy = oracle.round_bf16(np.array(DY, np.float64).reshape(-1))
    w = np.array(W, np.float32)
    out = {}
    y, r, _ = oracle.fwd(x, w, EPS, T, 1, H, H, H)
    out["plain.rstd"] = r
    out["plain.y"] = y.reshape(-1)
    out["plain.dx"] = oracle.bwd_dx(x, dy, r, w, T, 1, H, H, H).reshape(-1)
    out["plain.dw"] = oracle.bwd_dw(x, dy, r, T, 1, H, H, H)
    yr, rr, h = oracle.fwd(x, w, EPS, T, 1, H, H, H, residual=res)
    out["res.h_bits"] = h.reshape(-1).astype(np.float64)
    out["res.rstd"] = rr
    out["res.y"] = yr.reshape(-1)
    return out


def main():
    out = compute()
    with open(OUT, "w") as f:
        f.write("# FP64 oracle outputs for the typed-in inputs of make_golden.py\n")
        f.write("# (RMSNorm training forward/backward, flashinfer PR #8827 description).\n")
        f.write("# One line per tensor: name, then float.hex of each element.\n")
        for k, v in out.items():
            f.write(k + " " + " ".join(float(e).hex() for e in v) + "\n")
    print("wrote", OUT)


if __name__ == "__main__":
    main()
