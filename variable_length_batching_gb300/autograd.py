"""torch.autograd bindings of the block and of varlen attention, so that the
library's forward and backward calls can sit inside a training step
("DanLing NestedTensor" section 4.1 and Appendix A.1: the measured step is
forward, the sample-weighted loss and the backward).  Argument marshalling
only: the forward and the backward of each Function are the C-ABI calls of
``nt``.

    z_t, s_out = pair_block(part, s, W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g)
    o = varlen_attention(q, k, v, cu_seqlens, max_len)

``pair_block`` is the ReLU block of Eq. 1 on a square partition (the
forward: nt_pair_broadcast, nt_pair_transition, nt_pair_reduce; the
backward: nt_pair_block_backward, whose gradients are fp32 and are returned
in the dtype of each input).  ``varlen_attention`` is non-causal or causal
self-attention over cu_seqlens segments (the forward keeps the natural-log
LSE; the backward is nt_varlen_attn_bwd).
"""
from __future__ import annotations

from types import SimpleNamespace
from typing import Optional

import torch

from . import nt


class PairBlock(torch.autograd.Function):
    @staticmethod
    def forward(ctx, part, s, W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g, ln_eps):
        w = SimpleNamespace(W_a=W_a, W_b=W_b, ln_gamma=ln_gamma, ln_beta=ln_beta, W1=W1, b1=b1, W2=W2, b2=b2,
                            W_g=W_g, b_g=b_g)
        z_t, m, s_out = nt.block_forward(part, s, w, ln_eps=ln_eps)
        ctx.part = part
        ctx.ln_eps = ln_eps
        ctx.has_b = (b1 is not None, b2 is not None, b_g is not None)
        ctx.save_for_backward(s, W_a, W_b, ln_gamma, ln_beta, W1, b1 if b1 is not None else s.new_empty(0),
                              W2, b2 if b2 is not None else s.new_empty(0), W_g,
                              b_g if b_g is not None else s.new_empty(0), m)
        return z_t, s_out

    @staticmethod
    def backward(ctx, dz_t, ds_out):
        s, W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g, m = ctx.saved_tensors
        has_b1, has_b2, has_bg = ctx.has_b
        w = SimpleNamespace(W_a=W_a, W_b=W_b, ln_gamma=ln_gamma, ln_beta=ln_beta, W1=W1,
                            b1=b1 if has_b1 else None, W2=W2, b2=b2 if has_b2 else None, W_g=W_g,
                            b_g=b_g if has_bg else None)
        f32 = lambda t: None if t is None else t.float().contiguous()
        if ds_out is None:
            ds_out = torch.zeros(s.shape[0], W_g.shape[0], dtype=torch.float32, device=s.device)
        g = nt.nt_pair_block_backward(ctx.part, s, w, m, f32(ds_out), f32(dz_t), ln_eps=ctx.ln_eps)
        like = lambda grad, t: grad.to(t.dtype)
        return (None, like(g["ds"], s), like(g["dW_a"], W_a), like(g["dW_b"], W_b), like(g["dgamma"], ln_gamma),
                like(g["dbeta"], ln_beta), like(g["dW1"], W1), like(g["db1"], b1) if has_b1 else None,
                like(g["dW2"], W2), like(g["db2"], b2) if has_b2 else None, like(g["dW_g"], W_g),
                like(g["db_g"], b_g) if has_bg else None, None)


def pair_block(part: "nt.Partition", s: torch.Tensor, W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g,
               ln_eps: float = 1e-5):
    """The ReLU block of Eq. 1 with autograd: returns (z~, s_out)."""
    return PairBlock.apply(part, s, W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g, ln_eps)


class VarlenAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens, max_len, causal, scale):
        o, lse = nt.nt_varlen_attn_qk(q, k, v, cu_seqlens, cu_seqlens, max_len, scale=scale, causal=causal,
                                      want_lse=True)
        ctx.save_for_backward(q, k, v, o, lse, cu_seqlens)
        ctx.max_len, ctx.causal, ctx.scale = max_len, causal, scale
        return o

    @staticmethod
    def backward(ctx, d_o):
        q, k, v, o, lse, cu = ctx.saved_tensors
        dq, dk, dv = nt.nt_varlen_attn_bwd(q, k, v, o, d_o.to(q.dtype).contiguous(), lse, cu, None, ctx.max_len,
                                           scale=ctx.scale, causal=ctx.causal)
        return dq, dk, dv, None, None, None, None


def varlen_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor, max_len: int,
                     causal: bool = False, scale: Optional[float] = None):
    """Self-attention within each cu_seqlens segment, with autograd."""
    return VarlenAttention.apply(q, k, v, cu_seqlens, max_len, causal, scale)
