"""Drop-in fused linear cross-entropy loss for PyTorch autograd.

    loss = FusedLinearCrossEntropyLoss()(hidden_states, lm_head_weight, labels)
    loss.backward()

hidden_states [..., D] and lm_head_weight [V, D] are bfloat16 CUDA tensors,
labels [...] integer token ids (ignore_index marks ignored tokens). The call
replaces lm_head + cross-entropy (the interface the GPU MODE lecture 28 notes
show for the fused loss: hidden states (B*S, hidden), the LM-head weight
(vocab, hidden) and labels, replacing PyTorch's reduction="mean" loss) without
materialising the [N, V] logits.

As on the pages, the gradients are computed in the forward call (the logits
are recomputed tile by tile there, never stored); backward only multiplies
them by the upstream dL/dloss with the library's scaling kernel. Every
arithmetic step runs in libflce.so; this module only marshals tensors.
"""
from __future__ import annotations

import torch

from . import _binding as B


class FusedLinearCrossEntropyFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden_states, weight, labels, ignore_index: int, reduction: str):
        D = hidden_states.shape[-1]
        H = hidden_states.reshape(-1, D)
        if not H.is_contiguous():
            raise ValueError("hidden_states must be contiguous")
        y = labels.reshape(-1)
        if y.dtype != torch.int32:
            y = y.to(torch.int32)
        need_dh = ctx.needs_input_grad[0]
        need_dw = ctx.needs_input_grad[1]
        if reduction == "none" and (need_dh or need_dw):
            raise ValueError('reduction="none" has no backward here (it would need a per-token '
                             'upstream gradient)')
        if need_dh or need_dw:
            dw_dtype = "bfloat16" if weight.dtype == torch.bfloat16 else "float32"
            res = B.forward_backward(H, weight, y, need_dh=need_dh, need_dw=need_dw,
                                     ignore_index=ignore_index, reduction=reduction,
                                     dw_dtype=dw_dtype)
        else:
            res = B.forward(H, weight, y, ignore_index=ignore_index, reduction=reduction)
        ctx.hidden_shape = hidden_states.shape
        ctx.save_for_backward(res.dH, res.dW)
        loss = res.loss
        return loss.reshape(labels.shape) if reduction == "none" else loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        dH, dW = ctx.saved_tensors
        scale = grad_out.detach().reshape(1)
        if scale.dtype != torch.float32:
            scale = scale.to(torch.float32)
        B.scale_grads(dH, dW, scale.contiguous())
        dh = dH.reshape(ctx.hidden_shape) if dH is not None else None
        return dh, dW, None, None, None


class FusedLinearCrossEntropyLoss(torch.nn.Module):
    """nn.Module form: FusedLinearCrossEntropyLoss(ignore_index=-100,
    reduction="mean")(hidden_states, lm_head_weight, labels)."""

    def __init__(self, ignore_index: int = -100, reduction: str = "mean"):
        super().__init__()
        if reduction not in ("mean", "sum", "none"):
            raise ValueError(f"unsupported reduction {reduction!r}")
        self.ignore_index = int(ignore_index)
        self.reduction = reduction

    def forward(self, hidden_states, lm_head_weight, labels):
        return FusedLinearCrossEntropyFunction.apply(hidden_states, lm_head_weight, labels,
                                                     self.ignore_index, self.reduction)


def fused_linear_cross_entropy(hidden_states, lm_head_weight, labels, ignore_index: int = -100,
                               reduction: str = "mean"):
    """Functional form of FusedLinearCrossEntropyLoss."""
    return FusedLinearCrossEntropyFunction.apply(hidden_states, lm_head_weight, labels,
                                                 int(ignore_index), reduction)
