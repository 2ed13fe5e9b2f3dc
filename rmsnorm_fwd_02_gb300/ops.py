"""Torch-facing API: allocates outputs and workspace with torch, then calls the C ABI.

    y, rstd        = rmsnorm_fwd(x, w, eps)                  # x [T, H] or a [T, nh, H] view
    y, rstd, h     = rmsnorm_fwd(x_in, w, eps, residual=res) # fused residual add
    dx, dw         = rmsnorm_bwd(dy, x_or_h, rstd, w, deterministic=True, dh=None)
    dx, dw, rstd   = rmsnorm_bwd_recompute(dy, x_or_h, w, eps, deterministic=True, dh=None)
    y              = rmsnorm_train(x, w, eps, deterministic=True)   # autograd
    y              = rmsnorm_train(x, w, eps, recompute_rstd=True)  # saves x only
    y, h           = rmsnorm_train(x_in, w, eps, residual=res)      # autograd, residual form

Inputs: BF16 CUDA activations whose last dimension is contiguous (a [T, nh, H] view may
have any 16-byte-aligned token and head strides, e.g. the first 24 heads of a [T, 32*256]
buffer); w is BF16 or FP32 [H].  Outputs y, h, dx are contiguous BF16 of shape
[T, H] / [T, nh, H]; rstd is FP32 [T] / [T, nh]; dw is FP32 [H].
"""
from __future__ import annotations

import torch

from . import _native as N

EPS = 1e-6


def _view(x: torch.Tensor):
    if x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("activations must be CUDA bfloat16 tensors")
    if x.dim() == 2:
        T, H = x.shape
        if x.stride(1) != 1 and H > 1:
            raise ValueError("last dimension must be contiguous")
        return T, 1, H, x.stride(0) if T > 1 else H, H
    if x.dim() == 3:
        T, nh, H = x.shape
        if x.stride(2) != 1 and H > 1:
            raise ValueError("last dimension must be contiguous")
        s_tok = x.stride(0) if T > 1 else nh * H
        s_head = x.stride(1) if nh > 1 else H
        return T, nh, H, s_tok, s_head
    raise ValueError("activations must be [T, H] or [T, nh, H]")


def _wdtype(w: torch.Tensor) -> int:
    if w.dtype == torch.bfloat16:
        return N.RMSN_W_BF16
    if w.dtype == torch.float32:
        return N.RMSN_W_FP32
    raise TypeError("w must be bfloat16 or float32")


def rmsnorm_fwd(x, w, eps=EPS, residual=None):
    T, nh, H, s_tok, s_head = _view(x)
    if residual is not None:
        if residual.shape != x.shape or residual.stride() != x.stride():
            raise ValueError("residual must have x's shape and strides")
    w = w.contiguous()
    shape = (T, H) if x.dim() == 2 else (T, nh, H)
    y = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
    rstd = torch.empty(shape[:-1], dtype=torch.float32, device=x.device)
    h = torch.empty_like(y) if residual is not None else None
    N.rmsnorm_train_fwd(x, residual, w, _wdtype(w), y, h, rstd, T, nh, H, s_tok, s_head,
                        float(eps))
    return (y, rstd) if residual is None else (y, rstd, h)


def rmsnorm_bwd(dy, x, rstd, w, deterministic=True, dh=None):
    T, nh, H, s_tok, s_head = _view(x)
    dy = dy.contiguous()
    if dh is not None:
        dh = dh.contiguous()
    w = w.contiguous()
    dx = torch.empty(dy.shape, dtype=torch.bfloat16, device=dy.device)
    dw = torch.empty(H, dtype=torch.float32, device=dy.device)
    nbytes = N.rmsnorm_train_bwd_workspace_bytes(T, nh, H, deterministic)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dy.device)
    N.rmsnorm_train_bwd(x, dy, dh, rstd.contiguous(), w, _wdtype(w), dx, dw, ws, nbytes,
                        T, nh, H, s_tok, s_head, deterministic)
    return dx, dw


def rmsnorm_bwd_recompute(dy, x, w, eps=EPS, deterministic=True, dh=None):
    """The backward for a step that kept x but not rstd: rstd is recomputed from x inside
    the backward (and returned)."""
    T, nh, H, s_tok, s_head = _view(x)
    dy = dy.contiguous()
    if dh is not None:
        dh = dh.contiguous()
    w = w.contiguous()
    dx = torch.empty(dy.shape, dtype=torch.bfloat16, device=dy.device)
    dw = torch.empty(H, dtype=torch.float32, device=dy.device)
    rstd = torch.empty(dy.shape[:-1], dtype=torch.float32, device=dy.device)
    nbytes = N.rmsnorm_train_bwd_workspace_bytes(T, nh, H, deterministic)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dy.device)
    N.rmsnorm_train_bwd_recompute(x, dy, dh, w, _wdtype(w), dx, dw, rstd, ws, nbytes, T, nh, H,
                                  s_tok, s_head, float(eps), deterministic)
    return dx, dw, rstd


class RMSNormTrain(torch.autograd.Function):
    """Autograd wrapper: forward saves x (or h) and rstd -- or, with recompute_rstd, x (or
    h) alone, and the backward recomputes rstd; backward runs the CUDA backward."""

    @staticmethod
    def forward(ctx, x, w, eps, residual, deterministic, recompute_rstd):
        ctx.residual = residual is not None
        ctx.deterministic = deterministic
        ctx.recompute = recompute_rstd
        ctx.eps = eps
        if residual is None:
            y, rstd = rmsnorm_fwd(x, w, eps)
            xs = x
        else:
            y, rstd, xs = rmsnorm_fwd(x, w, eps, residual=residual)
        if recompute_rstd:
            ctx.save_for_backward(xs, w)
        else:
            ctx.save_for_backward(xs, rstd, w)
        return y if residual is None else (y, xs)

    @staticmethod
    def backward(ctx, *grads):
        if ctx.recompute:
            xs, w = ctx.saved_tensors
            rstd = None
        else:
            xs, rstd, w = ctx.saved_tensors
        dy = grads[0]
        dh = grads[1] if ctx.residual else None
        if dy is None:
            dy = torch.zeros(xs.shape, dtype=torch.bfloat16, device=xs.device)
        dy = dy.to(torch.bfloat16)
        dh = None if dh is None else dh.to(torch.bfloat16)
        if rstd is None:
            dx, dw, _ = rmsnorm_bwd_recompute(dy, xs, w, ctx.eps, ctx.deterministic, dh=dh)
        else:
            dx, dw = rmsnorm_bwd(dy, xs, rstd, w, ctx.deterministic, dh=dh)
        dw = dw.to(w.dtype)
        if ctx.residual:
            return dx, dw, None, dx, None, None
        return dx, dw, None, None, None, None


def rmsnorm_train(x, w, eps=EPS, residual=None, deterministic=True, recompute_rstd=False):
    return RMSNormTrain.apply(x, w, eps, residual, deterministic, recompute_rstd)
