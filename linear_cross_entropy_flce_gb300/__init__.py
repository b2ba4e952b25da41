"""Fused linear cross-entropy for GB300 (sm_103a).

The loss of a language-model head, mean over non-ignored tokens of
logsumexp(h_i W^T) - h_i . w_{y_i}, and its gradients dH and dW, computed by
hand-written tcgen05/TMA CUDA kernels without writing the [N, V] logits to
device memory. The C ABI is include/flce.h; this package is its Python binding.
"""
from ._binding import (FLCE_ERR_ALIGN, FLCE_ERR_CUDA, FLCE_ERR_DEVICE, FLCE_ERR_LABEL_RANGE,
                       FLCE_ERR_NULL, FLCE_ERR_OPTION, FLCE_ERR_SHAPE, FLCE_ERR_TIMEOUT,
                       FLCE_ERR_WORKSPACE, FLCE_OK, FLCEError, LIB_PATH, Options, Result,
                       ShardForward, backward_shard, ce_logits, check_status, forward,
                       forward_backward, forward_backward_fp8, forward_noalloc, forward_shard,
                       forward_workspace_size, get_plan, lib, make_options, noalloc_setup,
                       quantize_e4m3, scale_grads, status_string, workspace_size)
from .loss import (FusedLinearCrossEntropyFunction, FusedLinearCrossEntropyLoss,
                   fused_linear_cross_entropy)

__all__ = ["FLCE_ERR_ALIGN", "FLCE_ERR_CUDA", "FLCE_ERR_DEVICE", "FLCE_ERR_LABEL_RANGE",
           "FLCE_ERR_NULL", "FLCE_ERR_OPTION", "FLCE_ERR_SHAPE", "FLCE_ERR_TIMEOUT",
           "FLCE_ERR_WORKSPACE", "FLCE_OK", "FLCEError", "LIB_PATH", "Options", "Result",
           "ShardForward", "backward_shard", "ce_logits", "check_status", "forward",
           "forward_backward", "forward_backward_fp8", "forward_noalloc", "forward_shard",
           "forward_workspace_size", "get_plan", "lib", "make_options", "noalloc_setup",
           "quantize_e4m3", "scale_grads", "status_string", "workspace_size",
           "FusedLinearCrossEntropyFunction", "FusedLinearCrossEntropyLoss",
           "fused_linear_cross_entropy"]
