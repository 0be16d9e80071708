"""torch.autograd glue for the CUDA kernels: the forward saves (L, Q, K, V, O)
and the backward recomputes from them ("CS336 Assignment 2 notes" §1.4, the
FlashAttention-2 autograd function), so the kernels drop into a model in place
of its attention core ("CS324 lecture 8: 03_online_softmax_and_flash.py",
patched_model).  Argument marshalling only: every step runs in the library.
"""
from __future__ import annotations

import torch

from . import attention_backward, attention_forward


class FlashAttentionFunction(torch.autograd.Function):
    """O = softmax(Q K^T scale) V with the mask of fa_fwd_ex; bf16 CUDA tensors
    q [B,H,Nq,d], k, v [B,H,Nk,d].  Saves L (fp32 [B,H,Nq]), Q, K, V and O; no
    N x N tensor is kept."""

    @staticmethod
    def forward(ctx, q, k, v, causal: bool = False, scale=None, window: int = 0):
        q, k, v = (t.contiguous() for t in (q, k, v))
        o, lse = attention_forward(q, k, v, causal, scale, window)
        ctx.save_for_backward(lse, q, k, v, o)
        ctx.causal, ctx.scale, ctx.window = causal, scale, window
        return o

    @staticmethod
    def backward(ctx, do):
        lse, q, k, v, o = ctx.saved_tensors
        dq, dk, dv, _ = attention_backward(q, k, v, o, lse, do.contiguous(), ctx.causal, ctx.scale, ctx.window)
        return dq, dk, dv, None, None, None


def flash_attention(q, k, v, causal: bool = False, scale=None, window: int = 0):
    """Differentiable exact attention through the CUDA kernels."""
    return FlashAttentionFunction.apply(q, k, v, causal, scale, window)
