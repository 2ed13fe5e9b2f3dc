"""Seeded synthetic inputs for RMSNorm training.

This module only draws random numbers and stores them in the dtypes the op takes.  It
holds none of the op's arithmetic, and it is the one module that both the CUDA path's
tests/benchmark and the FP64 oracle read their inputs from, so both see the same bytes.

Recipes follow the five workloads the RMSNorm-training pages measure (flashinfer PR
#8827, description and Measurement: BF16 activations, BF16 or FP32 weight, eps 1e-6,
plain rows, the fused residual form at H=6144, per-head views [T,24,256] strided and
[T,4,256] contiguous with a shared w[256]):

* activations x (and residual, dy, dh): N(0, 1) drawn in FP32, rounded to BF16;
* the dw-stress family scales 1 % of the rows (picked by the same generator) by 16
  before the rounding;
* weights: 1 + 0.1 * N(0, 1) in FP32, rounded to BF16 where the workload's weight is BF16.

Draw order is fixed (x, residual, dy, dh, w, outlier rows) so that a case is a pure
function of its seed and sizes.  BF16 tensors are returned as numpy ``uint16`` bit
patterns; FP32 weights as ``float32``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

EPS = float(np.float32(1e-6))  # the FP32 eps the kernels receive, widened exactly


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 bit patterns through torch's round-to-nearest-even conversion."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _normal(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.standard_normal(n, dtype=np.float32)


@dataclass
class Case:
    """One seeded input set.  ``x`` (and ``residual``) are flat buffers addressed through
    the view (row (t, h) starts at t*s_tok + h*s_head); ``dy``/``dh`` are contiguous
    [T*nh, H]."""
    T: int
    nh: int
    H: int
    s_tok: int
    s_head: int
    x: np.ndarray
    dy: np.ndarray
    w: np.ndarray
    residual: np.ndarray | None = None
    dh: np.ndarray | None = None
    eps: float = EPS
    label: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return self.T * self.nh

    @property
    def w_fp32(self) -> bool:
        return self.w.dtype == np.float32


def make_case(seed: int, T: int, H: int, *, nh: int = 1, buf_heads: int | None = None,
              w_fp32: bool = False, residual: bool = False, dh: bool = False,
              outlier_frac: float = 0.0, outlier_scale: float = 16.0,
              label: str = "") -> Case:
    """Builds one case.

    ``buf_heads`` > ``nh`` makes a strided per-head view: the activation buffer is
    [T, buf_heads*H] and the view takes its first ``nh`` heads (s_tok = buf_heads*H,
    s_head = H).  Otherwise the view is contiguous (s_tok = nh*H, s_head = H)."""
    rng = np.random.default_rng(seed)
    bh = nh if buf_heads is None else buf_heads
    assert bh >= nh
    n_buf = T * bh * H
    n_out = T * nh * H
    xf = _normal(rng, n_buf)
    resf = _normal(rng, n_buf) if residual else None
    dyf = _normal(rng, n_out)
    dhf = _normal(rng, n_out) if dh else None
    wf = (1.0 + 0.1 * _normal(rng, H)).astype(np.float32)
    if outlier_frac > 0.0 and T > 0:
        n_out_rows = max(1, int(round(outlier_frac * T * nh)))
        rows = rng.choice(T * nh, size=n_out_rows, replace=False)
        # row r = (t, h) lives at t*s_tok + h*s_head in the buffer
        xv = xf.reshape(T, bh, H)
        xv[rows // nh, rows % nh, :] *= np.float32(outlier_scale)
    return Case(
        T=T, nh=nh, H=H, s_tok=bh * H, s_head=H,
        x=to_bf16_bits(xf),
        dy=to_bf16_bits(dyf),
        w=wf if w_fp32 else to_bf16_bits(wf),
        residual=None if resf is None else to_bf16_bits(resf),
        dh=None if dhf is None else to_bf16_bits(dhf),
        label=label,
    )


# ---- the five measured workloads -----------------------------------------------------

def tiny(seed: int = 0) -> Case:
    """T=64, H=256, FP32 weight, no residual."""
    return make_case(seed, 64, 256, w_fp32=True, label="tiny")


PLAIN_H = 4096
PLAIN_T = (1, 65, 1024, 4096, 16384, 65536)


def plain(T: int, seed: int = 0) -> Case:
    """Plain rows, H=4096, BF16 weight."""
    return make_case(seed, T, PLAIN_H, label=f"plain_T{T}_H{PLAIN_H}")


STRESS_H = (1536, 2048, 5120)
STRESS_T = (65, 4096, 32768, 65536, 98304, 131072)


def stress(T: int, H: int, seed: int = 0) -> Case:
    """dw-accuracy stress: 1 % of rows x16, FP32 weight."""
    return make_case(seed, T, H, w_fp32=True, outlier_frac=0.01,
                     label=f"stress_T{T}_H{H}" + (f"_seed{seed}" if seed else ""))


RES_H = 6144
RES_T = (1, 96, 7168, 30720, 65536)


def residual(T: int, seed: int = 0, with_dh: bool = False) -> Case:
    """Fused residual add, H=6144, BF16 weight."""
    return make_case(seed, T, RES_H, residual=True, dh=with_dh,
                     label=f"residual_T{T}_H{RES_H}")


HEAD_T = (64, 4096, 65536)


def heads_strided(T: int, seed: int = 0) -> Case:
    """[T,24,256] view of the first 24 heads of a [T, 32*256] buffer, FP32 w[256]."""
    return make_case(seed, T, 256, nh=24, buf_heads=32, w_fp32=True,
                     label=f"heads24of32_T{T}")


def heads_contig(T: int, seed: int = 0) -> Case:
    """[T,4,256] contiguous, FP32 w[256]."""
    return make_case(seed, T, 256, nh=4, w_fp32=True, label=f"heads4_T{T}")


# ---- LayerNorm beside it ----------------------------------------------------------------
#
# The normalization tables of ROCm TransformerEngine PR #478 benchmark LayerNorm on M rows
# of hidden_size in BF16 (M 1024..8192; hidden 3584, 4096, 8192 and 16384).  The pages give neither eps nor distributions: eps is 1e-5
# (the usual LayerNorm default) and the draws follow the RMSNorm recipe above, plus a bias
# 0.1 * N(0, 1) and, optionally, a per-row offset so that some rows have |mean| >> std.

LN_EPS = float(np.float32(1e-5))  # FP32, as the kernels receive it
LN_M = (1024, 2048, 4096, 8192)
LN_H = (3584, 4096, 8192, 16384)


@dataclass
class LnCase:
    """One seeded LayerNorm input set: x, dy BF16 [R, H]; w, b [H] (both BF16 or both
    FP32)."""
    R: int
    H: int
    x: np.ndarray
    dy: np.ndarray
    w: np.ndarray
    b: np.ndarray
    eps: float = LN_EPS
    label: str = ""

    @property
    def wb_fp32(self) -> bool:
        return self.w.dtype == np.float32


def make_ln_case(seed: int, R: int, H: int, *, wb_fp32: bool = False,
                 row_offset: float = 0.0, label: str = "") -> LnCase:
    """Draw order: x, dy, w, b, then (row_offset != 0) one offset per row, scaled by
    row_offset and added to that row of x before the rounding."""
    rng = np.random.default_rng(seed)
    xf = _normal(rng, R * H)
    dyf = _normal(rng, R * H)
    wf = (1.0 + 0.1 * _normal(rng, H)).astype(np.float32)
    bf = (0.1 * _normal(rng, H)).astype(np.float32)
    if row_offset != 0.0 and R > 0:
        off = (np.float32(row_offset) * _normal(rng, R)).astype(np.float32)
        xf = (xf.reshape(R, H) + off[:, None]).reshape(-1)
    return LnCase(
        R=R, H=H,
        x=to_bf16_bits(xf),
        dy=to_bf16_bits(dyf),
        w=wf if wb_fp32 else to_bf16_bits(wf),
        b=bf if wb_fp32 else to_bf16_bits(bf),
        label=label or f"layernorm_M{R}_H{H}",
    )
