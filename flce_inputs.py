"""Seeded synthetic inputs for fused linear cross-entropy (FLCE).

This module is shared by the CUDA path's tests and bench and by the CPU
oracle's tests. It holds no arithmetic of the method itself: it only draws
hidden states H, LM-head weights W and labels y, rounds the floating-point
draws to bfloat16 bit patterns (and widens them back), and places ignored
tokens. The FP8 variant's operand quantisation is part of what is checked, so
its reference lives in the oracle (oracle/e4m3.py), not here.

The workloads stand in for the language-model heads the Liger Kernel pages
discuss ("Liger Kernel: Fused Triton Kernels for LLM Training", section
"The Problem": B*S = 8192 tokens, hidden 4096, vocabulary 128256; the GPU MODE
lecture 28 notes, practice item 8: a 152K-vocabulary Qwen2 head). No dataset or
trained weights are used: every value is a seeded draw.

Recipe (the same for every workload):
  * one Philox counter-based stream per tensor, keyed by (seed, tensor id), so
    any tensor can be drawn without drawing the others;
  * H = round_bf16(h_scale * N(0,1)) and W = round_bf16(w_std * N(0,1)),
    drawn in float32, rounded to nearest-even bfloat16;
  * labels uniform over [0, V), or a Zipf(s) law truncated to ranks 1..V with
    P(rank r) proportional to r^-s, sampled by inverse CDF on float64
    cumulative weights; rank r is token id r-1;
  * exactly round(p_ignore * N) positions, picked by a seeded permutation, are
    set to ignore_index (-100).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

IGNORE_INDEX = -100

_STREAM_H, _STREAM_W, _STREAM_LABELS, _STREAM_IGNORE = 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int          # tokens (B*S)
    D: int          # hidden size
    V: int          # vocabulary size
    h_scale: float
    w_std: float
    labels: str     # "uniform" or "zipf"
    p_ignore: float
    zipf_s: float = 1.1
    seed: int = 0


# The five workloads: a tiny case the oracle finishes in well under a second,
# a Llama-2-like head, a Llama-3-8B-shaped head (B=2, S=4096), a Qwen2-7B-shaped
# head and a long-sequence stress case with peaked logits.
WORKLOADS = {
    "tiny": Workload("tiny", 64, 128, 1000, 1.0, 0.05, "uniform", 0.0),
    "llama2": Workload("llama2", 4096, 2048, 32000, 1.0, 0.02, "uniform", 0.05),
    "llama3_8b": Workload("llama3_8b", 8192, 4096, 128256, 1.0, 0.02, "zipf", 0.10),
    "qwen2_7b": Workload("qwen2_7b", 16384, 3584, 152064, 1.0, 0.02, "uniform", 0.0),
    "long_seq": Workload("long_seq", 32768, 4096, 128256, 2.0, 0.04, "zipf", 0.10),
}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to nearest-even bfloat16; return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    return bf16_bits_to_f32(b).astype(np.float64)


def normal_bf16(shape, scale: float, seed: int, stream: int, block_rows: int = 4096) -> np.ndarray:
    """bf16 bits of scale * N(0,1), drawn in float32 row blocks (bounded host memory)."""
    rows, cols = shape
    out = np.empty((rows, cols), dtype=np.uint16)
    g = _rng(seed, stream)
    s = np.float32(scale)
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        x = g.standard_normal((r1 - r0, cols), dtype=np.float32)
        if s != np.float32(1.0):
            x *= s
        out[r0:r1] = f32_to_bf16_bits(x)
    return out


def zipf_labels(n: int, V: int, s: float, g: np.random.Generator) -> np.ndarray:
    ranks = np.arange(1, V + 1, dtype=np.float64)
    w = ranks ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = g.random(n)
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, V - 1).astype(np.int32)


def make_labels(wl: Workload, N: Optional[int] = None) -> np.ndarray:
    N = wl.N if N is None else N
    g = _rng(wl.seed, _STREAM_LABELS)
    if wl.labels == "uniform":
        y = g.integers(0, wl.V, size=N, dtype=np.int64).astype(np.int32)
    elif wl.labels == "zipf":
        y = zipf_labels(N, wl.V, wl.zipf_s, g)
    else:
        raise ValueError(f"unknown label law {wl.labels!r}")
    k = int(round(wl.p_ignore * N))
    if k:
        pos = _rng(wl.seed, _STREAM_IGNORE).permutation(N)[:k]
        y[pos] = IGNORE_INDEX
    return y


def make_inputs(wl: Workload, N: Optional[int] = None):
    """Return (H bits uint16 [N,D], W bits uint16 [V,D], labels int32 [N]).

    N may be given to draw only a prefix-sized batch with the same laws (used
    for bounded CPU timing samples); with N=None the workload's own N is used.
    """
    N = wl.N if N is None else N
    H = normal_bf16((N, wl.D), wl.h_scale, wl.seed, _STREAM_H)
    W = normal_bf16((wl.V, wl.D), wl.w_std, wl.seed, _STREAM_W)
    y = make_labels(wl, N)
    return H, W, y


def get(name: str) -> Workload:
    return WORKLOADS[name]
