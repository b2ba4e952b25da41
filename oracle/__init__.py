"""CPU float64 oracle for fused linear cross-entropy: test infrastructure only.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
use it. The product path never imports it.
"""
from . import e4m3
from .flce_oracle import (IGNORE_INDEX, ce_logits, check_labels, flce, log_sum_exp_rows, logits_bytes,
                          logits_rows, sample_rows, sample_vocab)

__all__ = ["e4m3", "IGNORE_INDEX", "ce_logits", "check_labels", "flce", "log_sum_exp_rows", "logits_bytes",
           "logits_rows", "sample_rows", "sample_vocab"]
