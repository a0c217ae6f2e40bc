"""PyTorch autograd front end of the library: the head-chunked attention
layer, the sequence-tiled SwiGLU MLP and the tiled LM-head loss as
``torch.autograd.Function`` s and ``nn.Module`` s, so that a training loop
can use them in place of its own attention, MLP and loss.

Every forward and backward runs the library's kernels through the binding
(``upipe.py``); nothing here computes.  Weights are held as fp32 master
parameters: each call hands their bf16 rounding to the kernels and returns
the kernels' fp32 weight gradients, so no precision is lost in the gradient
sums.  Activations are bf16 CUDA tensors.
"""

from __future__ import annotations

import torch

from headwise_chunked_context_gb300 import upipe


# ------------------------------------------------------------------ attention

class _AttentionFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, wqkv, wo, cfg, keep):
        wqkv_b, wo_b = wqkv.to(torch.bfloat16), wo.to(torch.bfloat16)
        out, lse, kept = upipe.layer_forward(cfg, x.contiguous(), wqkv_b, wo_b, keep_o=keep)
        ctx.save_for_backward(x, wqkv_b, wo_b, lse)
        ctx.kept, ctx.cfg = kept, cfg
        return out

    @staticmethod
    def backward(ctx, dout):
        x, wqkv_b, wo_b, lse = ctx.saved_tensors
        dx, dwqkv, dwo = upipe.layer_backward(ctx.cfg, x.contiguous(), wqkv_b, wo_b,
                                              dout.to(torch.bfloat16).contiguous(), lse, ctx.kept)
        ctx.kept = None
        return dx, dwqkv, dwo, None, None


class HeadChunkedAttention(torch.nn.Module):
    """One GQA/RoPE causal attention layer computed U query heads at a time
    (upipe_attn_fwd / upipe_attn_bwd): ``out = Attention(x)`` for x [L, D]
    bf16.  keep: None (the backward recomputes each chunk's Q/K/V and O),
    "device_o" (O kept on the device) or "host" (O kept in page-locked host
    memory, the fastest)."""

    def __init__(self, D: int, H: int, Hkv: int, U: int, rope_theta: float = 500000.0, keep="host",
                 device="cuda", init_std: float = 0.02):
        super().__init__()
        self.D, self.H, self.Hkv, self.U, self.rope_theta = D, H, Hkv, U, rope_theta
        if keep not in (None, "device_o", "host"):
            raise ValueError(f"keep: expected None, 'device_o' or 'host', got {keep!r}")
        self.keep = {None: False, "device_o": True, "host": "host"}[keep]
        self.wqkv = torch.nn.Parameter(torch.randn((H + 2 * Hkv) * 128, D, device=device) * init_std)
        self.wo = torch.nn.Parameter(torch.randn(D, H * 128, device=device) * init_std)

    def forward(self, x):
        cfg = upipe.Config(L=x.shape[0], D=self.D, H=self.H, Hkv=self.Hkv, U=self.U, rope_theta=self.rope_theta)
        return _AttentionFn.apply(x, self.wqkv, self.wo, cfg, self.keep)


# ------------------------------------------------------------------- MLP

class _MlpFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, wgu, wd, T):
        wgu_b, wd_b = wgu.to(torch.bfloat16), wd.to(torch.bfloat16)
        y = upipe.mlp_forward(x.contiguous(), wgu_b, wd_b, T)
        ctx.save_for_backward(x, wgu_b, wd_b)
        ctx.T = T
        return y

    @staticmethod
    def backward(ctx, dy):
        x, wgu_b, wd_b = ctx.saved_tensors
        dx, dwgu, dwd = upipe.mlp_backward(x.contiguous(), wgu_b, wd_b, dy.to(torch.bfloat16).contiguous(), ctx.T)
        return dx, dwgu, dwd, None


class TiledSwiGLU(torch.nn.Module):
    """SwiGLU MLP computed T rows at a time (upipe_mlp_fwd / _bwd):
    ``y = (silu(x Wg^T) * (x Wu^T)) Wd^T`` for x [L, D] bf16; Wgu = [Wg; Wu]."""

    def __init__(self, D: int, F: int, T: int = 8192, device="cuda", init_std: float = 0.02):
        super().__init__()
        self.T = T
        self.wgu = torch.nn.Parameter(torch.randn(2 * F, D, device=device) * init_std)
        self.wd = torch.nn.Parameter(torch.randn(D, F, device=device) * init_std)

    def forward(self, x):
        return _MlpFn.apply(x, self.wgu, self.wd, self.T)


# ------------------------------------------------------------------- loss

class _CeFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, h, w, labels, T):
        valid = int((labels >= 0).sum())
        scale = 1.0 / max(1, valid)
        # loss and both gradients in one pass over the vocabulary, tile by tile
        loss, dh, dw = upipe.ce_loss(h.contiguous(), w.to(torch.bfloat16), labels.to(torch.int32).contiguous(),
                                     scale, T)
        ctx.save_for_backward(dh, dw)
        return loss.sum() * scale

    @staticmethod
    def backward(ctx, g):
        dh, dw = ctx.saved_tensors
        return (dh * g).to(torch.bfloat16), dw * g, None, None


class TiledCrossEntropy(torch.nn.Module):
    """Mean next-token cross-entropy of the LM head computed T rows at a time
    (upipe_ce_fwd_bwd): ``loss = mean_i logsumexp(h_i W^T) - (h_i W^T)[y_i]``
    over labels >= 0.  The gradients are formed together with the loss."""

    def __init__(self, D: int, V: int, T: int = 4096, device="cuda", init_std: float = 0.02):
        super().__init__()
        self.T = T
        self.w = torch.nn.Parameter(torch.randn(V, D, device=device) * init_std)

    def forward(self, h, labels):
        return _CeFn.apply(h, self.w, labels, self.T)


__all__ = ["HeadChunkedAttention", "TiledSwiGLU", "TiledCrossEntropy"]
