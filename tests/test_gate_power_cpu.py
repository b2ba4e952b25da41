"""The GPU parity gates can see the errors they exist for (CPU, no GPU).

A result with the precision the readings fix (G rounded once to bf16 from its
fp32 value, dW accumulated in fp32, dH rounded once to bf16) is built on the
host from the oracle's own lse, and must pass every gate of flce_testlib.
Mistakes are then planted in that host result, never in the CUDA path: a
softmax part 20% too small, the dW rows of ids that no token has as its label
set to zero, and the one-hot term moved to the wrong column. The pooled
Frobenius gate lets the first through (the one-hot term owns most of the
norm, and on the Llama-2-like head the rows of ids without hits hold 0.04% of
||dW||^2); the softmax-part and element-wise gates must stop all three."""
import types

import numpy as np
import pytest

import flce_inputs
import oracle
from flce_testlib import assert_within, compare

torch = pytest.importorskip("torch")


def _case():
    # the Llama-2-like head's weight scale (w_std 0.02) at a size the host handles in a second
    wl = flce_inputs.Workload("gate", 512, 256, 8000, 1.0, 0.02, "uniform", 0.05, seed=61)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H = flce_inputs.bf16_bits_to_f64(Hb)
    W = flce_inputs.bf16_bits_to_f64(Wb)
    ref = oracle.flce(H, W, y, want_abs=True)
    return H, W, y, ref


def _bf16(x):
    return flce_inputs.bf16_bits_to_f64(flce_inputs.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def _host_result(H, W, y, ref, softmax_factor=1.0, target_shift=0):
    """loss, lse, dH (bf16) and dW (fp32) with G = bf16(fl32(p * s)) off the target
    and bf16(fl32(-s * fl32(1 - p))) at it, as the fused path forms them. A
    target_shift plants the one-hot term in another column (subtracted there, the
    true target left at p * s)."""
    valid = y != -100
    s = np.float32(1.0 / valid.sum())
    p = np.exp(H @ W.T - ref["lse"][:, None]) * softmax_factor
    G = (p.astype(np.float32) * s).astype(np.float32)
    rows = np.nonzero(valid)[0]
    cols = (y[rows] + target_shift) % W.shape[0]
    if target_shift == 0:
        q = (-np.expm1(-ref["nll"][rows])).astype(np.float32)   # 1 - p of the target
        G[rows, cols] = (-np.float64(s) * q.astype(np.float64)).astype(np.float32)
    else:
        G[rows, cols] = (G[rows, cols] - s).astype(np.float32)
    G[~valid] = 0.0
    Gb = _bf16(G)
    dH = _bf16((Gb @ W).astype(np.float32))
    dW = (Gb.T @ H).astype(np.float32).astype(np.float64)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return types.SimpleNamespace(loss=t(np.array([ref["loss"]], dtype=np.float32)),
                                 lse=t(ref["lse"].astype(np.float32)),
                                 dH=t(dH.astype(np.float32)).to(torch.bfloat16), dW=t(dW))


def _errs(H, W, y, ref, res):
    return compare(res, ref, labels=y, Hg=H, Wg=W)


def test_result_at_the_stated_precision_passes():
    H, W, y, ref = _case()
    errs = _errs(H, W, y, ref, _host_result(H, W, y, ref))
    assert_within(errs)


def test_peaked_logits_at_the_stated_precision_pass():
    """The gates hold for the GPU test of peaked logits (std about 30, half of the
    labels on the row's largest logit): a result at the stated precision passes."""
    wl = flce_inputs.Workload("custom", 300, 256, 3000, 4.0, 0.5, "uniform", 0.05, seed=31)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H = flce_inputs.bf16_bits_to_f64(Hb)
    W = flce_inputs.bf16_bits_to_f64(Wb)
    top = np.argmax(H @ W.T, axis=1).astype(np.int32)
    half = np.arange(len(y)) % 2 == 0
    y = np.where((y != -100) & half, top, y).astype(np.int32)
    ref = oracle.flce(H, W, y, want_abs=True)
    errs = _errs(H, W, y, ref, _host_result(H, W, y, ref))
    assert_within(errs)


def test_target_entry_formed_from_the_fp32_lse_is_caught():
    """The arithmetic the fused path had before forming 1 - p in its merge: G from
    the fp32-rounded lse, the target entry as fl32(p * s) - s. On peaked logits
    (lse about 145) that entry carries half an lse ulp of the scale, far beyond
    itself for a confident token: the element-wise and per-row gates fail it."""
    wl = flce_inputs.Workload("custom", 300, 256, 3000, 4.0, 0.5, "uniform", 0.05, seed=31)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H = flce_inputs.bf16_bits_to_f64(Hb)
    W = flce_inputs.bf16_bits_to_f64(Wb)
    top = np.argmax(H @ W.T, axis=1).astype(np.int32)
    half = np.arange(len(y)) % 2 == 0
    y = np.where((y != -100) & half, top, y).astype(np.int32)
    ref = oracle.flce(H, W, y, want_abs=True)
    valid = y != -100
    s = np.float32(1.0 / valid.sum())
    lse32 = ref["lse"].astype(np.float32).astype(np.float64)
    G = (np.exp(H @ W.T - lse32[:, None]).astype(np.float32) * s).astype(np.float32)
    rows = np.nonzero(valid)[0]
    G[rows, y[rows]] = (G[rows, y[rows]] - s).astype(np.float32)
    G[~valid] = 0.0
    Gb = _bf16(G)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    res = types.SimpleNamespace(loss=t(np.array([ref["loss"]], dtype=np.float32)),
                                lse=t(ref["lse"].astype(np.float32)),
                                dH=t(_bf16((Gb @ W).astype(np.float32)).astype(np.float32)).to(torch.bfloat16),
                                dW=t((Gb.T @ H).astype(np.float32).astype(np.float64)))
    errs = _errs(H, W, y, ref, res)
    assert errs["dH_elem"] > 1.0 and errs["dW_elem"] > 1.0
    assert errs["dH_soft_row"] > 1.0 and errs["dW_soft_row"] > 1.0
    with pytest.raises(AssertionError):
        assert_within(errs)


def test_softmax_part_twenty_percent_off_is_caught():
    H, W, y, ref = _case()
    errs = _errs(H, W, y, ref, _host_result(H, W, y, ref, softmax_factor=0.8))
    assert errs["dW_fro"] <= 5e-3                                  # the pooled gate alone is blind
    assert errs["dW_soft"] > 1.0 and errs["dH_soft"] > 1.0
    with pytest.raises(AssertionError):
        assert_within(errs)


def test_zeroed_rows_of_ids_without_hits_are_caught():
    H, W, y, ref = _case()
    res = _host_result(H, W, y, ref)
    hit = np.zeros(W.shape[0], dtype=bool)
    hit[y[y != -100]] = True
    res.dW[torch.from_numpy(~hit)] = 0.0
    errs = _errs(H, W, y, ref, res)
    assert errs["dW_soft"] > 1.0 and errs["dW_soft_row"] > 1.0
    with pytest.raises(AssertionError):
        assert_within(errs)


def test_one_hot_in_the_wrong_column_is_caught():
    H, W, y, ref = _case()
    errs = _errs(H, W, y, ref, _host_result(H, W, y, ref, target_shift=1))
    assert errs["dW_elem"] > 1.0 and errs["dH_elem"] > 1.0
    with pytest.raises(AssertionError):
        assert_within(errs)
