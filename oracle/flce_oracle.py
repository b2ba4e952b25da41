"""CPU float64 oracle for fused linear cross-entropy (FLCE). TEST INFRASTRUCTURE.

This module is the correctness reference for the CUDA path. It is test
infrastructure only: the tests, the package's smoke check and the benchmark's
CPU-baseline leg may call it; the product path never does. It shares no code
with the CUDA path and imports nothing from the package.

What it computes (plain definition, one logits row per token, float64):
the language-model-head cross-entropy that Liger Kernel's fused linear
cross-entropy returns without materialising the logits.

  z_iv   = h_i . w_v                                   (logits, Z = H W^T)
  lse_i  = m_i + log sum_v exp(z_iv - m_i),  m_i = max_v z_iv
  l_i    = lse_i - z_{i,y_i}                           (per-token NLL)
  loss   = sum_{valid i} l_i / n     (mean)   or   sum_{valid i} l_i   (sum)
  g_iv   = (exp(z_iv - lse_i) - [v = y_i]) * grad_scale / n   (valid i; 0 otherwise)
  dH_i   = sum_v g_iv w_v          dW_v = sum_i g_iv h_i

Sources on the pages (Liger Kernel pages):
  * "Liger Kernel: Fused Triton Kernels for LLM Training", section "The
    Architecture", 1. Fused Linear Cross-Entropy with Online LogSumExp: the
    logits Z = H W^T and the stable form LSE(z) = m + log sum_j exp(z_j - m);
    immediate target-logit extraction.
  * same page, 2. In-Kernel Gradient Computation During the Backward Pass: the
    gradient softmax minus one-hot, dL/dH = (dL/dZ) W, dL/dW = (dL/dZ)^T H. The
    printed gradient formula is garbled (its denominator is identically 1 and it
    drops the 1/n of the mean); the page's own Python simulation, section
    "Implementation: Simulating Fused Linear Cross-Entropy in Python", applies
    the 1/N factor and subtracts 1 at the target, which is the reading taken.
  * GPU MODE lecture 28 notes, the cross-entropy section: the loss is a drop-in
    for PyTorch's cross entropy with reduction="mean".

Readings where the pages are silent:
  * tokens whose label equals ignore_index contribute nothing and are not
    counted in n (PyTorch's convention, which the pages' loss replaces);
  * n = 0 (every token ignored): loss 0 and zero gradients, no NaN;
  * a label outside [0, V) that is not ignore_index is an error.

Rows are independent, so the per-row quantities are computed over blocks of
rows only to bound host memory; blocking does not change any per-row result.
dW_v is a sum over all tokens; it is computed per block of vocabulary ids,
each column-block of G over all tokens at once, so no sum over tokens is split.

ce_logits() is the same loss over a given logits matrix (the unfused
cross-entropy that fused linear cross-entropy replaces).

Parity status: every function here is pinned by tests under tests/ (closed
forms, brute-force log-sum-exp, finite differences, the pages' printed
memory figures); none is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

IGNORE_INDEX = -100


def logits_rows(H: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z_iv = h_i . w_v in float64 for the given rows of H (Z = H W^T)."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def log_sum_exp_rows(Z: np.ndarray) -> np.ndarray:
    """Stable LSE per row: m + log(sum exp(z - m)), m = max z."""
    m = np.max(Z, axis=1)
    return m + np.log(np.sum(np.exp(Z - m[:, None]), axis=1))


def check_labels(labels: np.ndarray, V: int, ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    y = np.asarray(labels, dtype=np.int64)
    valid = y != ignore_index
    bad = valid & ((y < 0) | (y >= V))
    if np.any(bad):
        raise ValueError(f"label out of range at token {int(np.argmax(bad))}")
    return valid


def flce(H: np.ndarray, W: np.ndarray, labels: np.ndarray, *,
         ignore_index: int = IGNORE_INDEX, reduction: str = "mean",
         grad_scale: float = 1.0, normalizer: float = 0.0,
         dh_rows: Optional[Sequence[int]] = None, dw_rows: Optional[Sequence[int]] = None,
         want_grads: bool = True, row_block: int = 512, vocab_block: int = 4096,
         Hg: Optional[np.ndarray] = None, Wg: Optional[np.ndarray] = None,
         want_abs: bool = False) -> dict:
    """Loss, per-token LSE and gradients of fused linear cross-entropy, float64.

    H: [N, D], W: [V, D] (any real dtype; values are taken exactly in float64),
    labels: [N] integers. reduction "mean" divides by n = #valid tokens (or by
    `normalizer` when it is > 0), "sum" does not divide.

    dh_rows / dw_rows select which rows of dH (token ids) and dW (vocabulary ids)
    are computed; None means all.
    Hg / Wg (default H / W) are the operands of the two gradient products,
    dH = G Wg and dW = G^T Hg. The FP8 variant passes the dequantised FP8
    operands as H, W (they define the logits) and their bf16 originals as Hg, Wg. lse is always computed for every token because
    the loss and every dW row need all of them.
    want_abs also returns the same two products taken over magnitudes,
    dH_abs = |G| |Wg| and dW_abs = |G|^T |Hg| (rows as selected): the scale
    against which the rounding of each gradient element is measured (an
    element-wise error bound proportional to them holds even where the signed
    sums cancel).
    Returns dict(loss, lse[N], nll[N] (0 on ignored tokens), n_valid, dH, dW,
    dh_rows, dw_rows, dH_abs, dW_abs).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    Hg = H if Hg is None else np.asarray(Hg, dtype=np.float64)
    Wg = W if Wg is None else np.asarray(Wg, dtype=np.float64)
    N, D = H.shape
    V, D2 = W.shape
    if Hg.shape != H.shape or Wg.shape != W.shape:
        raise ValueError("gradient operands must match H and W in shape")
    if D != D2:
        raise ValueError("H and W disagree on the hidden size")
    if reduction not in ("mean", "sum"):
        raise ValueError(f"unsupported reduction {reduction!r}")
    valid = check_labels(labels, V, ignore_index)
    y = np.where(valid, np.asarray(labels, dtype=np.int64), 0)
    n_valid = int(np.count_nonzero(valid))

    if reduction == "sum":
        scale = grad_scale
    elif normalizer > 0:
        scale = grad_scale / normalizer
    else:
        scale = grad_scale / n_valid if n_valid > 0 else 0.0

    dh_sel = np.arange(N) if dh_rows is None else np.asarray(dh_rows, dtype=np.int64)
    dw_sel = np.arange(V) if dw_rows is None else np.asarray(dw_rows, dtype=np.int64)
    want_dh = np.zeros(N, dtype=bool)
    want_dh[dh_sel] = True

    lse = np.empty(N, dtype=np.float64)
    nll = np.zeros(N, dtype=np.float64)
    dH = np.zeros((len(dh_sel), D), dtype=np.float64) if want_grads else None
    dH_abs = np.zeros((len(dh_sel), D), dtype=np.float64) if (want_grads and want_abs) else None
    dh_pos = {int(r): k for k, r in enumerate(dh_sel)}

    # Pass over tokens: logits row, LSE, target logit, and dH for requested rows.
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Z = logits_rows(H[r0:r1], W)
        lse_b = log_sum_exp_rows(Z)
        lse[r0:r1] = lse_b
        rows = np.arange(r0, r1)
        zt = Z[rows - r0, y[r0:r1]]
        nll[r0:r1] = np.where(valid[r0:r1], lse_b - zt, 0.0)
        if want_grads:
            sel = rows[want_dh[r0:r1]]
            if len(sel):
                Zs = Z[sel - r0]
                G = np.exp(Zs - lse_b[sel - r0][:, None])
                G[np.arange(len(sel)), y[sel]] -= 1.0
                G *= scale
                G[~valid[sel]] = 0.0
                out = G @ Wg
                out_abs = np.abs(G) @ np.abs(Wg) if want_abs else None
                for k, r in enumerate(sel):
                    dH[dh_pos[int(r)]] = out[k]
                    if want_abs:
                        dH_abs[dh_pos[int(r)]] = out_abs[k]

    loss_sum = math.fsum(nll[valid].tolist())
    if reduction == "sum":
        loss = loss_sum
    elif normalizer > 0:
        loss = loss_sum / normalizer
    else:
        loss = loss_sum / n_valid if n_valid > 0 else 0.0

    dW = None
    dW_abs = None
    if want_grads:
        # Pass over vocabulary ids: the column block of G over all tokens, then
        # dW_v = sum_i g_iv h_i for every v in the block.
        dW = np.zeros((len(dw_sel), D), dtype=np.float64)
        if want_abs:
            dW_abs = np.zeros((len(dw_sel), D), dtype=np.float64)
        Hv = H[valid]
        Hgv = Hg[valid]
        yv = y[valid]
        lsev = lse[valid]
        for c0 in range(0, len(dw_sel), vocab_block):
            vids = dw_sel[c0:c0 + vocab_block]
            Zc = logits_rows(Hv, W[vids])                 # [n, |vids|]
            Gc = np.exp(Zc - lsev[:, None])
            Gc -= (yv[:, None] == vids[None, :])
            Gc *= scale
            dW[c0:c0 + len(vids)] = Gc.T @ Hgv
            if want_abs:
                dW_abs[c0:c0 + len(vids)] = np.abs(Gc).T @ np.abs(Hgv)

    return dict(loss=loss, lse=lse, nll=nll, n_valid=n_valid, dH=dH, dW=dW,
                dh_rows=dh_sel, dw_rows=dw_sel, dH_abs=dH_abs, dW_abs=dW_abs)


def ce_logits(Z: np.ndarray, labels: np.ndarray, *, ignore_index: int = IGNORE_INDEX,
              reduction: str = "mean", grad_scale: float = 1.0, normalizer: float = 0.0,
              want_grad: bool = True, row_block: int = 1024) -> dict:
    """Cross-entropy over given logits Z [N, V] (the unfused loss the fused one
    replaces: the cross-entropy section of the GPU MODE lecture 28 notes, which
    takes logits.view(-1, vocab) and labels with reduction="mean"), float64.

    Same definitions and readings as flce() with z_iv given directly:
    lse_i = m_i + log sum_v exp(z_iv - m_i), per-token loss lse_i - z_{i,y_i}
    (0 when ignored), loss = sum / n ("mean"), sum ("sum") or the per-token
    vector ("none"); dlogits = (exp(z - lse) - onehot) * grad_scale / n, zero rows
    for ignored tokens ("none" has no gradient here).
    Returns dict(loss, lse, nll, n_valid, dZ)."""
    Z = np.asarray(Z)
    N, V = Z.shape
    if reduction not in ("mean", "sum", "none"):
        raise ValueError(f"unsupported reduction {reduction!r}")
    valid = check_labels(labels, V, ignore_index)
    y = np.where(valid, np.asarray(labels, dtype=np.int64), 0)
    n_valid = int(np.count_nonzero(valid))
    if reduction == "sum":
        scale = grad_scale
    elif normalizer > 0:
        scale = grad_scale / normalizer
    else:
        scale = grad_scale / n_valid if n_valid > 0 else 0.0
    lse = np.empty(N, dtype=np.float64)
    nll = np.zeros(N, dtype=np.float64)
    dZ = np.zeros((N, V), dtype=np.float64) if (want_grad and reduction != "none") else None
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Zb = Z[r0:r1].astype(np.float64)
        lse_b = log_sum_exp_rows(Zb)
        lse[r0:r1] = lse_b
        k = np.arange(r1 - r0)
        nll[r0:r1] = np.where(valid[r0:r1], lse_b - Zb[k, y[r0:r1]], 0.0)
        if dZ is not None:
            G = np.exp(Zb - lse_b[:, None])
            G[k, y[r0:r1]] -= 1.0
            G *= scale
            G[~valid[r0:r1]] = 0.0
            dZ[r0:r1] = G
    total = math.fsum(nll[valid].tolist())
    if reduction == "none":
        loss = nll.copy()
    elif reduction == "sum":
        loss = total
    elif normalizer > 0:
        loss = total / normalizer
    else:
        loss = total / n_valid if n_valid > 0 else 0.0
    return dict(loss=loss, lse=lse, nll=nll, n_valid=n_valid, dZ=dZ)


def logits_bytes(N: int, V: int, elem_bytes: int = 4) -> int:
    """Bytes an unfused path holds for the [N, V] logits (fp32 by default):
    B*S*V*sizeof(float32), the formula of the page's section "The Problem"."""
    return int(N) * int(V) * int(elem_bytes)


def sample_rows(labels: np.ndarray, n_rows: int, seed: int, ignore_index: int = IGNORE_INDEX,
                n_ignored: int = 16, n_frequent_ids: int = 8) -> np.ndarray:
    """Token ids whose dH rows the sampled check uses: up to `n_ignored` ignored
    tokens, the tokens whose label is among the most frequent ids, and the rest
    uniform without replacement (seeded). Sorted, unique."""
    y = np.asarray(labels, dtype=np.int64)
    N = len(y)
    rng = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 77])))
    chosen = []
    ign = np.nonzero(y == ignore_index)[0]
    chosen.extend(ign[:n_ignored].tolist())
    valid_y = y[y != ignore_index]
    if len(valid_y):
        ids, counts = np.unique(valid_y, return_counts=True)
        top = ids[np.argsort(-counts, kind="stable")[:n_frequent_ids]]
        hits = np.nonzero(np.isin(y, top))[0]
        chosen.extend(hits[: max(0, n_rows // 4)].tolist())
    rest = np.setdiff1d(np.arange(N), np.asarray(chosen, dtype=np.int64))
    k = max(0, min(len(rest), n_rows - len(set(chosen))))
    chosen.extend(rng.choice(rest, size=k, replace=False).tolist())
    return np.unique(np.asarray(chosen, dtype=np.int64))


def sample_vocab(labels: np.ndarray, V: int, n_ids: int, seed: int,
                 ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """Vocabulary ids whose dW rows the sampled check uses: id V-1, up to half
    of `n_ids` taken from the most frequent label ids, the rest uniform over the
    remaining ids (seeded). Sorted, unique."""
    y = np.asarray(labels, dtype=np.int64)
    rng = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 78])))
    valid_y = y[y != ignore_index]
    chosen = {V - 1}
    if len(valid_y):
        ids, counts = np.unique(valid_y, return_counts=True)
        chosen.update(int(v) for v in ids[np.argsort(-counts, kind="stable")[: n_ids // 2]])
    rest = np.setdiff1d(np.arange(V), np.asarray(sorted(chosen), dtype=np.int64))
    k = max(0, min(len(rest), n_ids - len(chosen)))
    chosen.update(int(v) for v in rng.choice(rest, size=k, replace=False))
    return np.asarray(sorted(chosen), dtype=np.int64)
