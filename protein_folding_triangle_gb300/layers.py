"""Autograd functions and torch modules over the library's entry points.

Every computation runs in libtriattn's kernels; these classes only hold
parameters, keep the forward's context buffer
for the backward, and hand the library's gradients to autograd.  The
library's parameter gradients are FP32; autograd casts them to each
parameter's dtype (BF16 projection matrices, FP32 LayerNorm parameters).

- ``TriangleAttention``: the triangle-attention module around the core
  (LayerNorm, projections into q, k, v and the pair bias, core, output
  projection; "TurboPairFormer", Figure 6).  Returns the update; the caller
  adds it to z.
- ``TriangleMultiplication``: the triangle multiplicative update, outgoing or
  incoming ("TurboPairFormer", Figure 12).  Returns the update.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import triattn as T


class TriangleAttentionFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, z, ln_w, ln_b, w_in, w_o, mask, H: int, D: int):
        z = z.contiguous()
        out, buf = T.tri_attn_module_fwd(z, mask, ln_w, ln_b, w_in, w_o, H, D)
        ctx.save_for_backward(z, ln_w, w_in, w_o, buf)
        ctx.mask, ctx.H, ctx.D = mask, H, D
        return out

    @staticmethod
    def backward(ctx, d_out):
        z, ln_w, w_in, w_o, buf = ctx.saved_tensors
        dz, dlw, dlb, dwi, dwo = T.tri_attn_module_bwd(z, ctx.mask, ln_w, w_in, w_o, buf, d_out.contiguous(), ctx.H,
                                                       ctx.D)
        return dz, dlw, dlb, dwi, dwo, None, None, None


class TriangleMultiplicationFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, z, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, mask, direction: str):
        z = z.contiguous()
        out, buf = T.triattn_trimul_fwd(z, mask, ln_in_w, ln_in_b, w_p, ln_out_w, ln_out_b, w_o, direction)
        ctx.save_for_backward(z, ln_in_w, w_p, ln_out_w, w_o, buf)
        ctx.mask, ctx.direction = mask, direction
        return out

    @staticmethod
    def backward(ctx, d_out):
        z, ln_in_w, w_p, ln_out_w, w_o, buf = ctx.saved_tensors
        dz, dliw, dlib, dwp, dlow, dlob, dwo = T.triattn_trimul_bwd(z, ctx.mask, ln_in_w, w_p, ln_out_w, w_o, buf,
                                                                    d_out.contiguous(), ctx.direction)
        return dz, dliw, dlib, dwp, dlow, dlob, dwo, None, None


class TriangleAttention(torch.nn.Module):
    """Triangle attention over the pair tensor z [B, N, N, C] (BF16).  ``mask``
    (optional) is the core's additive key mask [B, N, N] (BF16, 0 or -inf):
    key k of slice i is masked where mask[b, i, k] = -inf."""

    def __init__(self, c_z: int, n_heads: int, head_dim: int, device=None):
        super().__init__()
        self.H, self.D = n_heads, head_dim
        f = 3 * n_heads * head_dim + n_heads
        self.ln_w = torch.nn.Parameter(torch.ones(c_z, dtype=torch.float32, device=device))
        self.ln_b = torch.nn.Parameter(torch.zeros(c_z, dtype=torch.float32, device=device))
        self.w_in = torch.nn.Parameter(
            (torch.randn(c_z, f, device=device) / math.sqrt(c_z)).to(torch.bfloat16))
        self.w_o = torch.nn.Parameter(
            (torch.randn(n_heads * head_dim, c_z, device=device) / math.sqrt(n_heads * head_dim)).to(torch.bfloat16))

    def forward(self, z: torch.Tensor, mask: Optional[torch.Tensor] = None) -> torch.Tensor:
        return TriangleAttentionFunction.apply(z, self.ln_w, self.ln_b, self.w_in, self.w_o, mask, self.H, self.D)


class TriangleMultiplication(torch.nn.Module):
    """Triangle multiplicative update of z [B, N, N, C_z] (BF16), ``direction``
    "outgoing" or "incoming".  ``mask`` (optional) is the multiplicative pair
    mask [B, N, N] (BF16, 1 keeps a pair)."""

    def __init__(self, c_z: int, c_hidden: int, direction: str = "outgoing", device=None):
        super().__init__()
        if direction not in T.TRIMUL_DIRECTIONS:
            raise ValueError(f"direction must be one of {tuple(T.TRIMUL_DIRECTIONS)}")
        self.direction = direction
        f = 4 * c_hidden + c_z
        self.ln_in_w = torch.nn.Parameter(torch.ones(c_z, dtype=torch.float32, device=device))
        self.ln_in_b = torch.nn.Parameter(torch.zeros(c_z, dtype=torch.float32, device=device))
        self.w_p = torch.nn.Parameter((torch.randn(c_z, f, device=device) / math.sqrt(c_z)).to(torch.bfloat16))
        self.ln_out_w = torch.nn.Parameter(torch.ones(c_hidden, dtype=torch.float32, device=device))
        self.ln_out_b = torch.nn.Parameter(torch.zeros(c_hidden, dtype=torch.float32, device=device))
        self.w_o = torch.nn.Parameter(
            (torch.randn(c_hidden, c_z, device=device) / math.sqrt(c_hidden)).to(torch.bfloat16))

    def forward(self, z: torch.Tensor, mask: Optional[torch.Tensor] = None) -> torch.Tensor:
        return TriangleMultiplicationFunction.apply(z, self.ln_in_w, self.ln_in_b, self.w_p, self.ln_out_w,
                                                    self.ln_out_b, self.w_o, mask, self.direction)
