"""torch.autograd integration: differential attention as a differentiable op.

``diff_attn(q1, k1, q2, k2, v, lam, lam_init, causal=False, gamma=None)``
runs the training forward (``fwd_train``) and, on ``backward``, the library's
backward pass (``bwd``); gradients flow to q1, k1, q2, k2, v, to lambda (a
learnable scalar on the Differential Transformer pages: the iloveeagents.com
Q&A, "Mathematical Formula") and to the GroupNorm gain gamma.  This module
only marshals tensors between autograd and the C ABI: every step runs in the
library's kernels.

lambda enters the C ABI as a host float, so a lambda held in a CUDA tensor
is read back to the host once per forward call (a stream synchronisation).
"""
from __future__ import annotations

import torch

from . import bwd, fwd_train


class DiffAttnFunction(torch.autograd.Function):
    """Inputs: q1, q2 [B,H,Nq,d], k1, k2 [B,H,Nk,d], v [B,H,Nk,dv] (CUDA bf16,
    contiguous); lam a 0-dim tensor or float; gamma a CUDA float32 [H*dv]
    tensor or None; lam_init, causal, eps plain values.  Output y [B,H,Nq,dv]
    bf16."""

    @staticmethod
    def forward(ctx, q1, k1, q2, k2, v, lam, gamma, lam_init, causal, eps):
        lam_f = float(lam.detach()) if isinstance(lam, torch.Tensor) else float(lam)
        y, saved = fwd_train(q1, k1, q2, k2, v, lam_f, lam_init, causal=causal, gamma=gamma, eps=eps)
        ctx.save_for_backward(q1, k1, q2, k2, v, saved["o_prenorm"], saved["o2"], saved["lse"],
                              gamma if gamma is not None else torch.empty(0, device=q1.device))
        ctx.has_gamma = gamma is not None
        ctx.lam, ctx.lam_init, ctx.causal, ctx.eps = lam_f, lam_init, causal, eps
        ctx.lam_is_tensor = isinstance(lam, torch.Tensor)
        ctx.lam_meta = (lam.shape, lam.dtype, lam.device) if ctx.lam_is_tensor else None
        return y

    @staticmethod
    def backward(ctx, dy):
        q1, k1, q2, k2, v, o_pre, o2, lse, gamma = ctx.saved_tensors
        gamma = gamma if ctx.has_gamma else None
        saved = {"o_prenorm": o_pre, "o2": o2, "lse": lse}
        g = bwd(q1, k1, q2, k2, v, dy.to(torch.bfloat16).contiguous(), saved, ctx.lam, ctx.lam_init,
                causal=ctx.causal, gamma=gamma, eps=ctx.eps)
        dlam = None
        if ctx.lam_is_tensor and ctx.needs_input_grad[5]:
            shape, dtype, device = ctx.lam_meta
            dlam = g["dlambda"].reshape(()).to(dtype=dtype, device=device).reshape(shape)
        dgamma = g["dgamma"] if (ctx.has_gamma and ctx.needs_input_grad[6]) else None
        return g["dq1"], g["dk1"], g["dq2"], g["dk2"], g["dv"], dlam, dgamma, None, None, None


def diff_attn(q1, k1, q2, k2, v, lam, lam_init, causal=False, gamma=None, eps=1e-5):
    """Differentiable DiffAttn + GroupNorm + (1 - lambda_init) scale; see
    ``DiffAttnFunction`` for shapes and types."""
    return DiffAttnFunction.apply(q1, k1, q2, k2, v, lam, gamma, lam_init, causal, eps)
