"""GPU parity of the vocabulary-shard calls (flce_forward_shard,
flce_backward_shard): the vocabulary is split into shards, each shard's
(m, s, zt) and gradient parts are computed on its own rows of W, and the
shards are combined the way a vocabulary-parallel caller's collective would
(max, rescaled sum, sum; then the sum of the fp32 dH parts and the
concatenation of the dW rows). The combination must give the float64 oracle's
loss, lse, dH and dW for the whole vocabulary."""
import types

import numpy as np
import pytest

import flce_inputs
import oracle
from flce_testlib import oracle_check, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import linear_cross_entropy_flce_gb300 as flce


def _combine(fwds):
    """The shards' combination in float64: M = max m, lse = M + log sum s exp(m - M),
    z_t = sum zt."""
    m = torch.stack([f.m for f in fwds]).double()
    s = torch.stack([f.s for f in fwds]).double()
    zt = torch.stack([f.zt for f in fwds]).double().sum(0)
    M = m.max(0).values
    return M + torch.log((s * torch.exp(m - M)).sum(0)), zt


def _run_shards(H, W, lab, bounds, V, fwd_opts=None, bwd_opts=None, reduction="mean"):
    fwd_opts, bwd_opts = fwd_opts or {}, bwd_opts or {}
    shards = list(zip(bounds[:-1], bounds[1:]))
    fwds = [flce.forward_shard(H, W[a:b], lab, a, V, **fwd_opts) for a, b in shards]
    for f in fwds:
        assert flce.check_status(f.status) == flce.FLCE_OK
    lse, zt = _combine(fwds)
    valid = lab != -100
    total = (lse - zt)[valid].sum()
    loss = total / valid.sum() if reduction == "mean" else total
    lse32 = lse.float().contiguous()
    dH = torch.zeros(H.shape, dtype=torch.float64, device=H.device)
    dWs = []
    for a, b in shards:
        r = flce.backward_shard(H, W[a:b], lab, lse32, a, V, reduction=reduction, **bwd_opts)
        assert flce.check_status(r.status) == flce.FLCE_OK
        assert r.dH.dtype == torch.float32
        dH += r.dH.double()
        dWs.append(r.dW)
    return types.SimpleNamespace(loss=loss.float(), lse=lse32, dH=dH, dW=torch.cat(dWs))


@pytest.mark.parametrize("bounds", [[0, 1000, 2300, 3000], [0, 256, 3000], [0, 2999, 3000]])
def test_vocabulary_shards_combine_to_the_oracle(bounds):
    N, D, V = 300, 256, 3000
    wl = flce_inputs.Workload("shards", N, D, V, 1.0, 0.05, "uniform", 0.07, seed=31)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    res = _run_shards(H, W, lab, bounds, V)
    ref = oracle.flce(flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb), y,
                      want_abs=True)
    oracle_check(res, Hb, Wb, y, ref, dh_f32=True, target_form="lse")


def test_whole_vocabulary_shard_softmax_part_in_fp32():
    """One shard holding the whole vocabulary returns dH in fp32, before any
    rounding to bf16, so the softmax part of dH is gated at 5e-3 with no output
    rounding in the budget: only G's one rounding per entry and fp32 sums. The
    Llama-2-like weight scale, several chunks and token blocks."""
    N, D, V = 1000, 512, 8000
    wl = flce_inputs.Workload("shard_whole", N, D, V, 1.0, 0.02, "uniform", 0.05, seed=34)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    plan = {"v_chunk": 2048, "n_block": 512}
    res = _run_shards(H, W, lab, [0, V], V, fwd_opts=plan, bwd_opts=plan)
    ref = oracle.flce(flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb), y,
                      want_abs=True)
    errs = oracle_check(res, Hb, Wb, y, ref, dh_f32=True, target_form="lse")
    assert errs["dH_soft_rel"] <= 5e-3


def test_shard_plans_sum_reduction_and_bf16_dw():
    """Several vocabulary chunks and token blocks inside a shard (its fp32 dH part
    stored by the first chunk and added to by the others), reduction "sum" with an
    upstream factor, bf16 dW rows."""
    N, D, V = 520, 200 + 56, 2600
    wl = flce_inputs.Workload("shards2", N, D, V, 1.0, 0.05, "zipf", 0.1, seed=32)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    plan = {"v_chunk": 512, "n_block": 256}
    res = _run_shards(H, W, lab, [0, 1300, 2600], V, fwd_opts=plan,
                      bwd_opts=dict(plan, grad_scale=0.5, dw_dtype="bfloat16"), reduction="sum")
    ref = oracle.flce(flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb), y,
                      reduction="sum", grad_scale=0.5, want_abs=True)
    oracle_check(res, Hb, Wb, y, ref, {"reduction": "sum", "grad_scale": 0.5,
                                       "dw_dtype": "bfloat16"}, dh_f32=True, target_form="lse")


def test_shard_label_outside_the_whole_vocabulary_sets_status():
    N, D, V = 64, 128, 1000
    wl = flce_inputs.Workload("shards3", N, D, V, 1.0, 0.05, "uniform", 0.0, seed=33)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    ok = flce.forward_shard(H, W[500:], lab, 500, V)   # labels below 500: other shards
    assert flce.check_status(ok.status) == flce.FLCE_OK
    lab[3] = V   # outside [0, V_total)
    bad = flce.forward_shard(H, W[500:], lab, 500, V)
    assert flce.check_status(bad.status) == flce.FLCE_ERR_LABEL_RANGE
