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

``q_up_proj_mxfp8(...)`` is the same layer with the MXFP8 query the pages'
module hands to attention (TransformerEngine PR "Add support for fused Q
Up-Proj GEMM/RoPE/Quant", flowchart: the fused up-projection emits an MXFP8
query, its scales go to the BHSD transpose and the GEMM swizzle, attention
may return a BF16 dQ). E4M3 codes and E8M0 scales are integer tensors that
autograd cannot differentiate, so the result is an ``Mxfp8Query``: the codes,
the scales (in the out_mode's layout) and an ``anchor``, a 0-d float tensor
that carries the graph. The consumer hands back the bf16 gradient of the
query with ``query.backward(dq)``; that runs this layer's backward, like
``q.backward(dq)`` on the bf16 face.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import bwd_dgrad, bwd_wgrad, fwd

__all__ = ["QUpProj", "q_up_proj", "Mxfp8Query", "q_up_proj_mxfp8"]


def _layer_backward(ctx, dq):
    """dx, dW, db of the layer for the upstream gradient dq [T, H, D] bf16,
    only those autograd asks for."""
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
        dW, db = bwd_wgrad(dq, x, cos, sin, H, Dn, Dr, pos=pos, db=ctx.has_bias and need_b, dq_pre_rope=rope)
    return dx if need_x else None, dW if need_w else None, db if need_b else None


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
        dx, dW, db = _layer_backward(ctx, dq)
        return dx, dW, db, None, None, None, None, None, None


def q_up_proj(x, W, cos, sin, H, Dn, Dr, bias=None, pos=None):
    """q = RoPE(x W^T + b) as bf16 [T, H, Dn + Dr], differentiable in x, W and b."""
    return QUpProj.apply(x, W, bias, cos, sin, pos, H, Dn, Dr)


class _GradBox:
    """Holds the query gradient the consumer hands in until the backward runs."""

    def __init__(self):
        self.dq = None


class _QUpProjMxfp8(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, W, bias, cos, sin, pos, H, Dn, Dr, out_mode, box):
        codes, scales = fwd(x, W, cos, sin, H, Dn, Dr, bias=bias, pos=pos, out_mode=out_mode)
        ctx.save_for_backward(x, W, cos, sin, pos)
        ctx.shape = (H, Dn, Dr)
        ctx.has_bias = bias is not None
        ctx.box = box
        ctx.mark_non_differentiable(codes, scales)
        anchor = torch.zeros((), dtype=torch.float32, device=x.device)
        return codes, scales, anchor

    @staticmethod
    def backward(ctx, g_codes, g_scales, g_anchor):
        dq = ctx.box.dq
        if dq is None:
            raise RuntimeError("the MXFP8 query's backward needs its bf16 gradient: call query.backward(dq)")
        ctx.box.dq = None
        dx, dW, db = _layer_backward(ctx, dq)
        return dx, dW, db, None, None, None, None, None, None, None, None


@dataclass
class Mxfp8Query:
    """The MXFP8 query of q_up_proj_mxfp8: codes uint8 [T, H, D] (E4M3),
    scales uint8 (E8M0; [T, H, ceil(D/32)] for out_mode "mxfp8", [H, T,
    ceil(D/32)] for "mxfp8_bhsd", each head in the GEMM's tiled order for
    "mxfp8_bhsd_swizzled"), and the anchor of the layer's autograd graph."""

    codes: torch.Tensor
    scales: torch.Tensor
    anchor: torch.Tensor
    _box: _GradBox

    def backward(self, dq: torch.Tensor) -> None:
        """Run the layer's backward for the query gradient dq (bf16 [T, H, D],
        e.g. the BF16 dQ of attention): dx, dW and db accumulate into the
        inputs' .grad like any autograd backward."""
        if dq.dtype != torch.bfloat16 or tuple(dq.shape) != tuple(self.codes.shape):
            raise ValueError(f"dq must be bf16 {list(self.codes.shape)}, got {dq.dtype} {list(dq.shape)}")
        self._box.dq = dq
        self.anchor.backward()


def q_up_proj_mxfp8(x, W, cos, sin, H, Dn, Dr, bias=None, pos=None, out_mode="mxfp8") -> Mxfp8Query:
    """The layer with an MXFP8 query (out_mode "mxfp8", "mxfp8_bhsd" or
    "mxfp8_bhsd_swizzled"), differentiable in x, W and b through
    Mxfp8Query.backward(dq)."""
    if out_mode not in ("mxfp8", "mxfp8_bhsd", "mxfp8_bhsd_swizzled"):
        raise ValueError(f"out_mode must be an MXFP8 mode, got {out_mode!r}")
    box = _GradBox()
    codes, scales, anchor = _QUpProjMxfp8.apply(x, W, bias, cos, sin, pos, H, Dn, Dr, out_mode, box)
    return Mxfp8Query(codes, scales, anchor, box)
