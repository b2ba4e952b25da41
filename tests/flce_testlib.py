"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C ABI, and compare with the CPU oracle.

Gates (each written out in assert_within):
  * loss relative 1e-3, per-token lse absolute 2e-3, dH and dW relative
    Frobenius 5e-3 (the numerics gate);
  * the softmax part of the gradients. In dH and in the dW rows of label ids the
    one-hot term (-scale at each token's target) dominates the norm (about 94%
    of ||dH|| and 98% of ||dW|| on the Llama-2-like head), so the pooled
    Frobenius gate cannot see an error in exp(z - lse) * scale. The softmax part
    is the gradient minus each token's target-entry contribution c_i x_i, where
    c_i = g_{i,y_i} = scale * (p_i - 1), p_i = exp(-nll_i) and x_i is w_{y_i} (dH)
    or h_i (dW row y_i). From the oracle the exact c_i is removed; from the GPU
    result the value that the precision reading admits for that entry: G is
    rounded once to bf16 from its fp32 value, and at the target that rounding is
    as large as the whole softmax part of a row. The fused path forms that fp32
    value as -scale * (1 - p) from the forward merge's 1 - p (no cancellation
    when p is close to 1); a vocabulary shard's backward, which has only lse, as
    p * scale - scale. What is left compares
    sum over non-target entries of g_iv x: relative Frobenius <= 5e-3 over the
    rows (per group of dW ids at full size), <= 2e-2 per row (plus 1e-6 of the
    largest row: a row whose whole gradient is below that, a token so confident
    that its gradient is about 1e-17, is zero at the output's precision). Outputs rounded to
    bf16 (dH always, dW on request) add their own rounding, whose root-mean-square
    is at most 2^-8/sqrt(3) of the output's norm; that amount is added to the
    bound (aggregate and per row). So is the fp32 accumulation of sums that the
    one-hot terms dominate (a dW row of an id with many hits, where the softmax
    part can be 1e-4 of the row): each of the K additions (K = tokens for dW,
    vocabulary ids for dH) rounds at 2^-24 of the running sum, a random walk of
    about 2^-24 sqrt(K) of the output's norm; the bound adds 2^-22 sqrt(K) of it
    (four times that: the tensor cores' adders need not round to nearest);
  * element-wise, |gpu - oracle| <= RHO * (|G||W|) (dH) or RHO * (|G|^T|H|) (dW),
    plus 2^-8 * (|ref| + RHO * that) for bf16 outputs, plus a floor of 1e-6 of
    the largest magnitude product. RHO = 2^-8 (one bf16 rounding of each G
    entry) + 2e-3 (relative error of p allowed by the lse tolerance) + 1e-3 (fp32
    accumulation). Magnitude products instead of |ref| keep the bound valid
    where the signed sums cancel.
"""
from __future__ import annotations

import itertools

import numpy as np

import flce_inputs

TOL_LOSS_REL = 1e-3
TOL_LSE_ABS = 2e-3
TOL_GRAD_FRO = 5e-3
TOL_SOFT_FRO = 5e-3
TOL_SOFT_ROW = 2e-2
U_BF16 = 2.0 ** -8                 # unit roundoff of bfloat16 (8 significant bits)
NOISE_BF16 = U_BF16 / np.sqrt(3.0)  # upper estimate of the rms relative rounding error
ACC_F32 = 2.0 ** -22                # per sqrt(addition): fp32 accumulation noise allowance
RHO = U_BF16 + 2e-3 + 1e-3
# per-row gates: rows whose whole gradient is below 1e-6 of the largest row are
# zero at the output's precision (the element-wise bound has the same floor)
ROW_FLOOR = 1e-6
IGNORE_INDEX = -100


def to_device(Hb, Wb, y, dev="cuda:0"):
    import torch
    H = torch.from_numpy(np.ascontiguousarray(Hb).view(np.int16)).to(dev).view(torch.bfloat16)
    W = torch.from_numpy(np.ascontiguousarray(Wb).view(np.int16)).to(dev).view(torch.bfloat16)
    lab = torch.from_numpy(np.ascontiguousarray(y, dtype=np.int32)).to(dev)
    return H, W, lab


def bf16_tensor_to_f64(t) -> np.ndarray:
    import torch
    return flce_inputs.bf16_bits_to_f64(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def tensor_to_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_tensor_to_f64(t)
    return t.double().cpu().numpy()


def rel_fro(a, b) -> float:
    nb = float(np.linalg.norm(b))
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def grad_scale_f32(n_valid: int, opts: dict | None = None) -> np.float32:
    """The factor of G as the reduction defines it (grad_scale / n for "mean",
    grad_scale / normalizer with a normalizer, grad_scale for "sum"), rounded to
    fp32 as the library holds it."""
    o = opts or {}
    gs = float(np.float32(o.get("grad_scale", 1.0)))
    if o.get("reduction", "mean") == "sum":
        return np.float32(gs)
    norm = float(np.float32(o.get("normalizer", 0.0)))
    if norm > 0:
        return np.float32(gs / norm)
    return np.float32(gs / n_valid) if n_valid > 0 else np.float32(0.0)


def _bf16_round(x32: np.ndarray) -> np.ndarray:
    return flce_inputs.bf16_bits_to_f64(flce_inputs.f32_to_bf16_bits(np.asarray(x32, dtype=np.float32)))


def target_terms(nll: np.ndarray, valid: np.ndarray, scale32: np.float32, scale64: float,
                 form: str = "ratio"):
    """Per token: the oracle's target entry c = scale * (p - 1) with p = exp(-nll),
    and the bf16 value(s) the GPU's G can hold there, rounded once to bf16 from
    its fp32 value. form "ratio" (the fused path, which keeps 1 - p = q from the
    forward merge): fl32(-s * fl32(q)); form "lse" (a vocabulary shard's backward,
    which has only lse): fl32(fl32(p * s) - s). Where a relative error of 1e-4 in
    q (or p) or two fp32 ulps of s could move the fp32 value across a bf16
    rounding boundary, both neighbours are admissible (alt is NaN elsewhere).
    Ignored tokens: 0."""
    nll = np.asarray(nll, dtype=np.float64)
    p = np.exp(-nll)
    s32 = np.float32(scale32)
    c_exact = np.where(valid, scale64 * (p - 1.0), 0.0)
    if form == "ratio":
        q = -np.expm1(-nll)                      # 1 - p without cancellation
        x = q * np.float64(s32)
        mid = np.float32(-np.float64(np.float32(q)) * np.float64(s32))
        lo = np.float32(-x * (1.0 + 1e-4) - 2.0 * np.spacing(np.float32(x)))
        hi = np.float32(-x * (1.0 - 1e-4) + 2.0 * np.spacing(np.float32(x)))
    elif form == "lse":
        ulp = np.float64(np.spacing(s32))
        x = p * np.float64(s32)
        mid = np.float32(np.float32(np.float32(p) * s32) - s32)
        lo = np.float32((x * (1.0 + 1e-4)) - np.float64(s32) - 2.0 * ulp)
        hi = np.float32((x * (1.0 - 1e-4)) - np.float64(s32) + 2.0 * ulp)
    else:
        raise ValueError(form)
    c_gpu = _bf16_round(mid)
    b_lo, b_hi = _bf16_round(lo), _bf16_round(hi)
    alt = np.where(b_lo != c_gpu, b_lo, np.where(b_hi != c_gpu, b_hi, np.nan))
    c_gpu = np.where(valid, c_gpu, 0.0)
    alt = np.where(valid, alt, np.nan)
    return c_exact, c_gpu, alt


def _best_rows(delta, alt_terms):
    """delta: [rows, D] differences; alt_terms: list of (row, vector) alternatives
    (adding the vector gives the other admissible rounding of one target entry).
    For each affected row pick the combination with the smallest norm."""
    by_row = {}
    for r, vec in alt_terms:
        by_row.setdefault(r, []).append(vec)
    n_combos = 0
    for r, vecs in by_row.items():
        vecs = vecs[:8]   # more than eight boundary cases in one row does not occur
        best = delta[r].copy()
        for mask in itertools.product([0, 1], repeat=len(vecs)):
            cand = delta[r] + sum(v for v, m in zip(vecs, mask) if m) if any(mask) else delta[r]
            n_combos += 1
            if np.linalg.norm(cand) < np.linalg.norm(best):
                best = cand
        delta[r] = best
    return len(by_row)


def _ratio(num, den):
    if num == 0.0:
        return 0.0
    return float(num / den) if den > 0 else float("inf")


def compare(res, ref, dh_rows=None, dw_rows=None, *, labels=None, Hg=None, Wg=None, opts=None,
            dh_f32=False, dw_groups=None, target_form="ratio") -> dict:
    """Errors of a GPU result against the oracle's.

    res: the binding's result (loss, lse, dH, dW tensors); ref: oracle.flce(...),
    with want_abs=True for the element-wise bound. dh_rows / dw_rows (device index
    tensors) select the GPU rows matching ref["dh_rows"] / ref["dw_rows"].
    labels, Hg, Wg (host arrays: the gradient operands, float32 or float64) and
    opts (reduction, grad_scale, normalizer, ignore_index, dw_dtype) enable the
    softmax-part gates. dh_f32: dH is fp32 (not rounded to bf16). dw_groups maps a
    name to positions in ref["dw_rows"] that are gated separately. target_form:
    how the GPU formed G's target entry (target_terms)."""
    o = opts or {}
    ignore = o.get("ignore_index", IGNORE_INDEX)
    dw_bf16 = o.get("dw_dtype") == "bfloat16"
    loss = float(res.loss.item())
    lse = res.lse.double().cpu().numpy()
    out = {"loss_gpu": loss, "loss_ref": ref["loss"]}
    out["loss_rel"] = abs(loss - ref["loss"]) / max(abs(ref["loss"]), 1e-30) if ref["loss"] else abs(loss)
    out["lse_abs"] = float(np.max(np.abs(lse - ref["lse"])))
    soft = labels is not None
    if soft:
        y = np.asarray(labels, dtype=np.int64)
        valid = y != ignore
        s32 = grad_scale_f32(ref["n_valid"], o)
        s64 = _scale64(ref["n_valid"], o)
        c_exact, c_gpu, c_alt = target_terms(ref["nll"], valid, s32, s64, target_form)
        yc = np.where(valid, y, 0)

    if getattr(res, "dH", None) is not None and ref["dH"] is not None:
        dH = tensor_to_f64(res.dH if dh_rows is None else res.dH[dh_rows])
        dref = ref["dH"]
        out["dH_fro"] = rel_fro(dH, dref)
        rows = ref["dh_rows"]
        if soft and Wg is not None:
            Wy = np.asarray(Wg[yc[rows]], dtype=np.float64)
            delta = dH - dref - (c_gpu[rows] - c_exact[rows])[:, None] * Wy
            amb = np.nonzero(np.isfinite(c_alt[rows]))[0]
            out["dH_boundary_rows"] = _best_rows(
                delta, [(k, -(c_alt[rows][k] - c_gpu[rows][k]) * Wy[k]) for k in amb])
            t_ref = dref - c_exact[rows][:, None] * Wy
            noise = (0.0 if dh_f32 else NOISE_BF16) + ACC_F32 * np.sqrt(Wg.shape[0])
            nu = noise * float(np.linalg.norm(dref))
            out["dH_soft_rel"] = rel_fro(delta + t_ref, t_ref)
            out["dH_soft"] = _ratio(float(np.linalg.norm(delta)),
                                    TOL_SOFT_FRO * float(np.linalg.norm(t_ref)) + nu)
            dn = np.linalg.norm(delta, axis=1)
            rn = np.linalg.norm(dref, axis=1)
            den = (TOL_SOFT_ROW * np.linalg.norm(t_ref, axis=1) + noise * rn
                   + ROW_FLOOR * float(rn.max(initial=0.0)))
            live = den > 0
            out["dH_soft_row"] = float(np.max(dn[live] / den[live])) if np.any(live) else 0.0
            if np.any(~live & (dn > 0)):
                out["dH_soft_row"] = float("inf")
        if ref.get("dH_abs") is not None:
            A = ref["dH_abs"]
            bound = RHO * A + (0.0 if dh_f32 else U_BF16 * (np.abs(dref) + RHO * A)) + 1e-6 * float(A.max(initial=0.0))
            err = np.abs(dH - dref)
            out["dH_elem"] = float(np.max(np.where(err > 0, err / np.maximum(bound, 1e-300), 0.0), initial=0.0))

    if getattr(res, "dW", None) is not None and ref["dW"] is not None:
        dW = tensor_to_f64(res.dW if dw_rows is None else res.dW[dw_rows])
        dref = ref["dW"]
        vids = ref["dw_rows"]
        groups = dw_groups or {"all": np.arange(len(vids))}
        for name, g in groups.items():
            key = "dW_fro" if name == "all" else f"dW_fro[{name}]"
            out[key] = rel_fro(dW[g], dref[g])
        if soft and Hg is not None:
            V = int(max(int(vids.max()) + 1, int(y.max(initial=0)) + 1))
            pos = np.full(V, -1, dtype=np.int64)
            pos[vids] = np.arange(len(vids))
            toks = np.nonzero(valid & (pos[yc] >= 0))[0]
            Hh = np.asarray(Hg[toks], dtype=np.float64)
            corr = np.zeros_like(dref)
            oneh = np.zeros_like(dref)
            np.add.at(corr, pos[yc[toks]], (c_gpu[toks] - c_exact[toks])[:, None] * Hh)
            np.add.at(oneh, pos[yc[toks]], c_exact[toks][:, None] * Hh)
            delta = dW - dref - corr
            amb = [k for k in range(len(toks)) if np.isfinite(c_alt[toks[k]])]
            out["dW_boundary_rows"] = _best_rows(
                delta, [(int(pos[yc[toks[k]]]), -(c_alt[toks[k]] - c_gpu[toks[k]]) * Hh[k]) for k in amb])
            t_ref = dref - oneh
            noise = (NOISE_BF16 if dw_bf16 else 0.0) + ACC_F32 * np.sqrt(len(y))
            for name, g in groups.items():
                sfx = "" if name == "all" else f"[{name}]"
                nu = noise * float(np.linalg.norm(dref[g]))
                out["dW_soft_rel" + sfx] = rel_fro(delta[g] + t_ref[g], t_ref[g])
                out["dW_soft" + sfx] = _ratio(float(np.linalg.norm(delta[g])),
                                              TOL_SOFT_FRO * float(np.linalg.norm(t_ref[g])) + nu)
                dn = np.linalg.norm(delta[g], axis=1)
                rn = np.linalg.norm(dref[g], axis=1)
                den = (TOL_SOFT_ROW * np.linalg.norm(t_ref[g], axis=1) + noise * rn
                       + ROW_FLOOR * float(rn.max(initial=0.0)))
                live = den > 0
                r = float(np.max(dn[live] / den[live])) if np.any(live) else 0.0
                out["dW_soft_row" + sfx] = float("inf") if np.any(~live & (dn > 0)) else r
        if ref.get("dW_abs") is not None:
            A = ref["dW_abs"]
            bound = RHO * A + (U_BF16 * (np.abs(dref) + RHO * A) if dw_bf16 else 0.0) + 1e-6 * float(A.max(initial=0.0))
            err = np.abs(dW - dref)
            out["dW_elem"] = float(np.max(np.where(err > 0, err / np.maximum(bound, 1e-300), 0.0), initial=0.0))
    return out


def _scale64(n_valid: int, opts: dict) -> float:
    """The oracle's (float64) factor of G for the same options."""
    gs = float(np.float32(opts.get("grad_scale", 1.0)))
    if opts.get("reduction", "mean") == "sum":
        return gs
    norm = float(np.float32(opts.get("normalizer", 0.0)))
    if norm > 0:
        return gs / norm
    return gs / n_valid if n_valid > 0 else 0.0


def assert_within(errs: dict):
    assert errs["loss_rel"] <= TOL_LOSS_REL, errs
    assert errs["lse_abs"] <= TOL_LSE_ABS, errs
    for k, v in errs.items():
        if k.startswith("dH_fro") or k.startswith("dW_fro"):
            assert v <= TOL_GRAD_FRO, (k, errs)
        elif k.startswith(("dH_soft", "dW_soft", "dH_elem", "dW_elem")) and "_rel" not in k:
            assert v <= 1.0, (k, errs)


def dw_sample_groups(y, vids, V, n_frequent=32):
    """Positions in vids of the three kinds of sampled vocabulary ids, gated apart:
    id V-1, the most frequent label ids, and the uniform picks (mostly ids that no
    token has as its label, whose dW row is all softmax part)."""
    ids, counts = np.unique(y[y != -100], return_counts=True)
    top = set(int(v) for v in ids[np.argsort(-counts, kind="stable")[:n_frequent]])
    groups = {"last": [], "frequent": [], "uniform": []}
    for k, v in enumerate(vids):
        key = "last" if v == V - 1 else "frequent" if int(v) in top else "uniform"
        groups[key].append(k)
    return {k: np.asarray(g, dtype=np.int64) for k, g in groups.items() if g}


def oracle_check(res, Hb, Wb, y, ref, opts=None, **kw) -> dict:
    """compare() with the bf16 inputs as the gradient operands, then assert_within."""
    errs = compare(res, ref, labels=y, Hg=flce_inputs.bf16_bits_to_f64(Hb),
                   Wg=flce_inputs.bf16_bits_to_f64(Wb), opts=opts, **kw)
    print(errs)
    assert_within(errs)
    return errs
