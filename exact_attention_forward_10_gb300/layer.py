"""A causal self-attention layer whose attention core is ``fattn_fwd``.

The drop-in use the pages walk through ("FlashAttention-2 in an attention
layer": the kernel replaces the QK^T / softmax / PV part of an attention
layer; the projections stay ordinary PyTorch).  Input ``x`` is
``[B, T, d_model]``; one fused projection gives Q, K and V for ``heads``
heads of ``d_model // heads`` columns (64, 128 or 256), the kernel computes
causal attention on ``[B, heads, T, head_dim]`` tensors, and an output
projection maps back to ``d_model``.

Nothing of size T x T is ever allocated: beyond the projections' activations
the attention call adds only O (the size of Q) and the fp32 LSE.
"""
from __future__ import annotations

import math

import torch
from torch import nn

from . import forward as _attention


class ExactAttention(nn.Module):
    """Causal multi-head self-attention with the fused exact-attention kernel.

    Weights are ordinary ``nn.Linear`` parameters (no bias), created in the
    module's dtype; the layer runs in fp16 or bf16 on a CUDA device.
    """

    def __init__(self, d_model: int, heads: int, causal: bool = True,
                 device=None, dtype=None) -> None:
        super().__init__()
        if d_model % heads:
            raise ValueError("d_model must be a multiple of heads")
        self.heads = heads
        self.head_dim = d_model // heads
        if self.head_dim not in (64, 128, 256):
            raise ValueError("head_dim (d_model / heads) must be 64, 128 or 256")
        self.causal = causal
        self.qkv = nn.Linear(d_model, 3 * d_model, bias=False, device=device, dtype=dtype)
        self.out = nn.Linear(d_model, d_model, bias=False, device=device, dtype=dtype)

    def split_heads(self, x: torch.Tensor):
        """Project ``x`` and return Q, K, V as contiguous [B, heads, T, head_dim]."""
        B, T, _ = x.shape
        qkv = self.qkv(x).view(B, T, 3, self.heads, self.head_dim)
        return tuple(qkv[:, :, i].transpose(1, 2).contiguous() for i in range(3))

    def merge_heads(self, o: torch.Tensor) -> torch.Tensor:
        B, H, T, D = o.shape
        return self.out(o.transpose(1, 2).reshape(B, T, H * D))

    def forward(self, x: torch.Tensor, return_lse: bool = False):
        q, k, v = self.split_heads(x)
        o, lse = _attention(q, k, v, causal=self.causal,
                            scale=1.0 / math.sqrt(self.head_dim))
        y = self.merge_heads(o)
        return (y, lse) if return_lse else y


def score_matrix_bytes(B: int, heads: int, T: int, dtype_bytes: int = 2) -> int:
    """Bytes of the T x T score matrices a materialising layer holds at once."""
    return dtype_bytes * B * heads * T * T


def attention_state_bytes(B: int, heads: int, T: int, head_dim: int,
                          dtype_bytes: int = 2) -> int:
    """Bytes the fused attention call writes besides its inputs: O (same size
    as Q) and the fp32 LSE.  The running (m, l) and the unnormalised O live
    in registers and TMEM on the chip and never reach device memory."""
    return B * heads * T * (head_dim * dtype_bytes + 4)
