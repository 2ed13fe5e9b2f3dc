"""Torch-facing LayerNorm API: allocates outputs and workspace with torch, then calls the
C ABI (include/layernorm_train.h).

    y, mean, rstd  = layernorm_fwd(x, w, b, eps)                 # x [..., H] contiguous
    dx, dw, db     = layernorm_bwd(dy, x, mean, rstd, w, deterministic=True)
    y              = layernorm_train(x, w, b, eps)                # autograd

Inputs: BF16 CUDA activations, contiguous, last dimension H (every leading dimension is a
row); w and b are both BF16 or both FP32 [H].  Outputs y, dx have x's shape (BF16); mean
and rstd are FP32 with x's leading shape; dw, db are FP32 [H].
"""
from __future__ import annotations

import torch

from . import _native as N

EPS = 1e-5


def _rows(x: torch.Tensor):
    if x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("activations must be CUDA bfloat16 tensors")
    if x.dim() < 1 or not x.is_contiguous():
        raise ValueError("activations must be contiguous with the row in the last dimension")
    H = x.shape[-1]
    return x.numel() // H if H else 0, H


def _wbdtype(w: torch.Tensor, b: torch.Tensor | None = None) -> int:
    if b is not None and b.dtype != w.dtype:
        raise TypeError("w and b must have the same dtype")
    if w.dtype == torch.bfloat16:
        return N.RMSN_W_BF16
    if w.dtype == torch.float32:
        return N.RMSN_W_FP32
    raise TypeError("w and b must be bfloat16 or float32")


def layernorm_fwd(x, w, b, eps=EPS):
    R, H = _rows(x)
    w = w.contiguous()
    b = b.contiguous()
    y = torch.empty_like(x)
    mean = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    rstd = torch.empty_like(mean)
    N.layernorm_train_fwd(x, w, b, _wbdtype(w, b), y, mean, rstd, R, H, float(eps))
    return y, mean, rstd


def layernorm_bwd(dy, x, mean, rstd, w, deterministic=True):
    R, H = _rows(x)
    dy = dy.contiguous()
    w = w.contiguous()
    dx = torch.empty_like(x)
    dw = torch.empty(H, dtype=torch.float32, device=x.device)
    db = torch.empty(H, dtype=torch.float32, device=x.device)
    nbytes = N.layernorm_train_bwd_workspace_bytes(R, H, deterministic)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    N.layernorm_train_bwd(x, dy, mean.contiguous(), rstd.contiguous(), w, _wbdtype(w), dx, dw,
                          db, ws, nbytes, R, H, deterministic)
    return dx, dw, db


class LayerNormTrain(torch.autograd.Function):
    """Autograd wrapper: forward saves x, mean and rstd; backward runs the CUDA backward."""

    @staticmethod
    def forward(ctx, x, w, b, eps, deterministic):
        y, mean, rstd = layernorm_fwd(x, w, b, eps)
        ctx.save_for_backward(x, mean, rstd, w)
        ctx.deterministic = deterministic
        ctx.b_dtype = b.dtype
        return y

    @staticmethod
    def backward(ctx, dy):
        x, mean, rstd, w = ctx.saved_tensors
        dx, dw, db = layernorm_bwd(dy.to(torch.bfloat16).contiguous(), x, mean, rstd, w,
                                   ctx.deterministic)
        return dx, dw.to(w.dtype), db.to(ctx.b_dtype), None, None


def layernorm_train(x, w, b, eps=EPS, deterministic=True):
    return LayerNormTrain.apply(x, w, b, eps, deterministic)
