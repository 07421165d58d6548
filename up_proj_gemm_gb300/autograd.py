"""Autograd face of the fused query up-projection (argument marshalling only).

TransformerEngine PR "Add a backwards linear function to be used with the
fused mla q up-proj": the layer is a PyTorch autograd function whose
backward runs the RoPE backward and then the linear backward with the saved
input. Megatron-LM PR "Fix fused MLA YaRN RoPE query kernel corrupting
upstream tensor in-place", discussion: the weight gradient uses the linear's
saved input x, not its output.

``q_up_proj(x, W, cos, sin, H, Dn, Dr, bias=None, pos=None)`` returns
q [T, H, Dn + Dr] bf16 = RoPE(x W^T + b). Its backward calls the library's
dgrad and wgrad entry points; dgrad hands the rotated rope channels to
wgrad. Only the gradients autograd asks for are computed. Every step runs in
the library's CUDA kernels; this module only moves tensors.
"""
from __future__ import annotations

import torch

from . import bwd_dgrad, bwd_wgrad, fwd

__all__ = ["QUpProj", "q_up_proj"]


class QUpProj(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, W, bias, cos, sin, pos, H, Dn, Dr):
        q = fwd(x, W, cos, sin, H, Dn, Dr, bias=bias, pos=pos, out_mode="bf16")
        ctx.save_for_backward(x, W, cos, sin, pos)
        ctx.shape = (H, Dn, Dr)
        ctx.has_bias = bias is not None
        return q

    @staticmethod
    def backward(ctx, dq):
        x, W, cos, sin, pos = ctx.saved_tensors
        H, Dn, Dr = ctx.shape
        need_x, need_w, need_b = ctx.needs_input_grad[0], ctx.needs_input_grad[1], ctx.needs_input_grad[2]
        dq = dq.contiguous()
        dx = dW = db = None
        rope = None
        if need_x:
            # dgrad also stores the rotated rope channels when wgrad follows
            if need_w or need_b:
                rope = torch.empty((x.shape[0], H, Dr), dtype=torch.bfloat16, device=dq.device)
            dx = bwd_dgrad(dq, W, cos, sin, H, Dn, Dr, pos=pos, dq_pre_rope=rope)
        if need_w or need_b:
            dW, db = bwd_wgrad(dq, x, cos, sin, H, Dn, Dr, pos=pos, db=ctx.has_bias and need_b,
                               dq_pre_rope=rope)
        return (dx if need_x else None, dW if need_w else None, db if need_b else None,
                None, None, None, None, None, None)


def q_up_proj(x, W, cos, sin, H, Dn, Dr, bias=None, pos=None):
    """q = RoPE(x W^T + b) as bf16 [T, H, Dn + Dr], differentiable in x, W and b."""
    return QUpProj.apply(x, W, bias, cos, sin, pos, H, Dn, Dr)
