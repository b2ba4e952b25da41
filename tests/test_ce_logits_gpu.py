"""GPU parity of the cross-entropy over given logits (flce_ce_logits) against
the CPU float64 oracle's ce_logits, with the numerics gate of the fused path
(loss rel 1e-3, lse abs 2e-3, gradient relative Frobenius 5e-3) and, because the
one-hot entries own most of that norm, an element-wise bound on every gradient
entry: |gpu - oracle| <= rho * (|ref| + 2 scale [v = y]) + 1e-37, rho = the
output's rounding (2^-8 for bf16, 2^-22 for fp32, the exponential's error) plus
2e-3 (the relative error of p that the lse tolerance allows); scale (p + [v = y])
bounds the entry's magnitude, and 1e-37 covers exponentials below 2^-126 that
the GPU flushes to zero."""
import numpy as np
import pytest

import flce_inputs
import oracle
from flce_testlib import grad_scale_f32, rel_fro, tensor_to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import linear_cross_entropy_flce_gb300 as flce


def _logits(N, V, seed, std=1.3, ld=None, bf16=False, p_ignore=0.05):
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 91])))
    Z = (g.standard_normal((N, V), dtype=np.float32) * np.float32(std))
    if bf16:
        Z = flce_inputs.bf16_bits_to_f32(flce_inputs.f32_to_bf16_bits(Z))
    y = g.integers(0, V, N).astype(np.int32)
    k = int(round(p_ignore * N))
    if k:
        y[g.permutation(N)[:k]] = -100
    ld = ld or V
    dev = torch.device("cuda:0")
    full = torch.zeros(N, ld, dtype=torch.float32)
    full[:, :V] = torch.from_numpy(Z)
    t = full.to(dev)
    if bf16:
        t = t.to(torch.bfloat16)
    return Z.astype(np.float64), y, t[:, :V], torch.from_numpy(y).to(dev)


def _check(res, ref, grad=True, per_token=False, y=None, opts=None):
    if per_token:
        assert np.max(np.abs(res.loss.double().cpu().numpy() - ref["loss"])) <= 2e-3
    else:
        loss = float(res.loss.item())
        assert abs(loss - ref["loss"]) <= 1e-3 * max(abs(ref["loss"]), 1e-30)
    assert np.max(np.abs(res.lse.double().cpu().numpy() - ref["lse"])) <= 2e-3
    if grad:
        d = tensor_to_f64(res.dlogits)
        err = rel_fro(d, ref["dZ"])
        assert err <= 5e-3, err
        if y is not None:
            r = ref["dZ"]
            onehot = np.zeros(r.shape, dtype=bool)
            rows = np.nonzero(np.asarray(y) != (opts or {}).get("ignore_index", -100))[0]
            onehot[rows, np.asarray(y)[rows]] = True
            sc = abs(float(grad_scale_f32(ref["n_valid"], opts)))
            rho = (2.0 ** -8 if res.dlogits.dtype == torch.bfloat16 else 2.0 ** -22) + 2e-3
            bound = rho * (np.abs(r) + 2.0 * sc * onehot) + 1e-37
            worst = float(np.max(np.abs(d - r) / bound))
            assert worst <= 1.0, worst


@pytest.mark.parametrize("N,V,ld", [(333, 5003, 5004), (1, 3, 4), (64, 4096, 4096), (257, 32000, 32008)])
def test_fp32_logits_parity(N, V, ld):
    Z, y, t, lab = _logits(N, V, seed=N + V, ld=ld)
    res = flce.ce_logits(t, lab)
    assert flce.check_status(res.status) == flce.FLCE_OK
    _check(res, oracle.ce_logits(Z, y), y=y)


@pytest.mark.parametrize("N,V", [(200, 32000), (77, 1001)])
def test_bf16_logits_parity(N, V):
    ld = (V + 7) // 8 * 8
    Z, y, t, lab = _logits(N, V, seed=N * 3 + V, bf16=True, ld=ld)
    res = flce.ce_logits(t, lab)
    assert flce.check_status(res.status) == flce.FLCE_OK
    _check(res, oracle.ce_logits(Z, y), y=y)


def test_in_place_equals_out_of_place():
    for bf16 in (False, True):
        Z, y, t, lab = _logits(300, 12000, seed=41, bf16=bf16)
        a = flce.ce_logits(t.clone(), lab)
        tc = t.clone()
        b = flce.ce_logits(tc, lab, in_place=True)
        torch.cuda.synchronize()
        assert b.dlogits.data_ptr() == tc.data_ptr()
        assert torch.equal(a.dlogits.view(torch.int16 if bf16 else torch.int32),
                           b.dlogits.view(torch.int16 if bf16 else torch.int32))
        assert torch.equal(a.loss, b.loss) and torch.equal(a.lse, b.lse)


@pytest.mark.parametrize("opts", [{"reduction": "sum"}, {"grad_scale": 3.0}, {"normalizer": 500.0}])
def test_reductions_and_scales(opts):
    Z, y, t, lab = _logits(150, 2048, seed=42, p_ignore=0.2)
    res = flce.ce_logits(t, lab, **opts)
    _check(res, oracle.ce_logits(Z, y, **opts), y=y, opts=opts)


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("grad_scale", [-2.5, 0.75])
def test_staged_rows_with_scales_and_ignored_tokens(bf16, grad_scale):
    """Rows long enough for the shared-memory staged kernel (bf16: 131 KB rows,
    fp32: 262 KB rows, both on clusters of 3 CTAs), a fifth of the tokens ignored,
    and a negative or fractional upstream gradient scale: the bf16 gradient pass
    takes the scale's magnitude into the exponent and applies its sign to the
    packed result, so both signs are checked element by element."""
    N, V = 48, 65600
    ld = (V + 7) // 8 * 8
    Z, y, t, lab = _logits(N, V, seed=47 + int(bf16), bf16=bf16, ld=ld, p_ignore=0.2)
    opts = {"grad_scale": grad_scale}
    res = flce.ce_logits(t, lab, **opts)
    assert flce.check_status(res.status) == flce.FLCE_OK
    _check(res, oracle.ce_logits(Z, y, **opts), y=y, opts=opts)
    ignored = torch.from_numpy(y == -100).to(t.device)
    assert int(ignored.sum()) > 0
    assert torch.count_nonzero(res.dlogits[ignored]).item() == 0


@pytest.mark.parametrize("N,V,bf16", [(64, 5003, False), (64, 40000, False), (48, 65600, True)])
def test_confident_targets_keep_their_small_gradient(N, V, bf16):
    """Logits with a standard deviation of 20 and half of the labels on the row's
    largest logit, so p of those targets is close to 1: the gradient at the
    target, scale * (p - 1), and the per-token loss, -log p, are small numbers
    that a difference with the fp32 lse would lose. Both must match the oracle
    to the output's own precision (1e-4 relative for fp32, one bf16 rounding for
    bf16), on the streamed kernel (20 KB rows) and the staged one."""
    ld = (V + 7) // 8 * 8
    Z, y, t, lab = _logits(N, V, seed=48 + V % 7, std=20.0, ld=ld, bf16=bf16, p_ignore=0.1)
    top = np.argmax(Z, axis=1).astype(np.int32)
    half = np.arange(N) % 2 == 0
    y = np.where((y != -100) & half, top, y).astype(np.int32)
    lab = torch.from_numpy(y).to(t.device)
    ref = oracle.ce_logits(Z, y)
    res = flce.ce_logits(t, lab)
    assert flce.check_status(res.status) == flce.FLCE_OK
    _check(res, ref, y=y)
    rows = np.nonzero(y != -100)[0]
    g = tensor_to_f64(res.dlogits)[rows, y[rows]]
    c = ref["dZ"][rows, y[rows]]
    rel = (2.0 ** -8) if bf16 else 1e-4
    # the float64 reference itself forms p - 1 with a cancellation: below 1e-12 of
    # the scale its own rounding takes over (a difference with the fp32 lse would
    # be off by about 1e-6 of the scale)
    floor = 1e-12 * abs(float(grad_scale_f32(ref["n_valid"])))
    assert np.all(np.abs(g - c) <= rel * np.abs(c) + floor), float(np.max(np.abs(g - c) / np.abs(c)))
    per = flce.ce_logits(t, lab, need_grad=False, reduction="none")
    nll = per.loss.double().cpu().numpy()
    want = ref["nll"]
    assert np.all(np.abs(nll - want) <= 1e-4 * np.abs(want) + 1e-6)


def test_per_token_losses_forward_only():
    Z, y, t, lab = _logits(150, 2048, seed=43, p_ignore=0.2)
    res = flce.ce_logits(t, lab, need_grad=False, reduction="none")
    _check(res, oracle.ce_logits(Z, y, reduction="none"), grad=False, per_token=True)


def test_large_magnitude_logits_are_stable():
    Z, y, t, lab = _logits(64, 3000, seed=44, std=40.0)
    res = flce.ce_logits(t, lab)
    assert torch.isfinite(res.dlogits).all()
    _check(res, oracle.ce_logits(Z, y), y=y)


def test_label_edges_and_all_ignored():
    Z, y, t, lab = _logits(128, 1000, seed=45, p_ignore=0.0)
    y[:40] = 0
    y[40:80] = 999
    lab = torch.from_numpy(y).to(t.device)
    _check(flce.ce_logits(t, lab), oracle.ce_logits(Z, y), y=y)
    y[:] = -100
    lab = torch.from_numpy(y).to(t.device)
    res = flce.ce_logits(t, lab)
    assert float(res.loss.item()) == 0.0 and torch.count_nonzero(res.dlogits).item() == 0
    y[5] = 1000
    lab = torch.from_numpy(y).to(t.device)
    res = flce.ce_logits(t, lab)
    assert flce.check_status(res.status) == flce.FLCE_ERR_LABEL_RANGE


def test_matches_fused_loss_on_the_same_logits():
    """The unfused loss over Z = H W^T (computed here in float64 and rounded to
    fp32) agrees with the fused loss of (H, W) within the numerics gate."""
    wl = flce_inputs.Workload("ce_vs_flce", 256, 512, 4000, 1.0, 0.05, "uniform", 0.1, seed=46)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    Hd, Wd = flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb)
    Z = (Hd @ Wd.T).astype(np.float32)
    dev = torch.device("cuda:0")
    ce = flce.ce_logits(torch.from_numpy(Z).to(dev), torch.from_numpy(y).to(dev))
    from flce_testlib import to_device
    fu = flce.forward(*to_device(Hb, Wb, y))
    torch.cuda.synchronize()
    assert abs(float(ce.loss.item()) - float(fu.loss.item())) <= 1e-4 * float(fu.loss.item())
    assert float((ce.lse - fu.lse).abs().max()) <= 1e-3


@pytest.mark.parametrize("N,V,bf16", [
    (40, 128256, False),   # 501 KB rows: staged slices, cluster of 5
    (24, 128257, True),    # 250 KB bf16 rows with a scalar tail: staged, cluster of 5
    (1000, 65600, True),   # bf16, cluster of 3, about 10 rows per cluster: both buffers
                           # and both exchange slots reused many times
    (400, 128257, True),   # bf16 with a tail, cluster of 5, about 7 rows per cluster
    (9, 100003, False),    # staged (cluster of 4), ragged fp32 tail
    (4, 240007, False),    # 938 KB rows: streamed kernel, cluster of 4
])
def test_long_rows_parity_and_in_place(N, V, bf16):
    """Rows long enough for multi-CTA clusters (shared-memory staged slices, or
    the streamed kernel past 768 KB): parity with the oracle, and the in-place
    gradient bitwise equal to the out-of-place one (the target logit must be read
    before any CTA of the cluster overwrites its slice)."""
    ld = (V + 7) // 8 * 8
    Z, y, t, lab = _logits(N, V, seed=N + V % 997, bf16=bf16, ld=ld)

    def padded_clone(x):  # same padded row stride (16-byte aligned rows)
        full = torch.zeros(N, ld, dtype=x.dtype, device=x.device)
        full[:, :V].copy_(x)
        return full[:, :V]

    a = flce.ce_logits(padded_clone(t), lab)
    assert flce.check_status(a.status) == flce.FLCE_OK
    _check(a, oracle.ce_logits(Z, y), y=y)
    tc = padded_clone(t)
    b = flce.ce_logits(tc, lab, in_place=True)
    torch.cuda.synchronize()
    assert flce.check_status(b.status) == flce.FLCE_OK
    assert b.dlogits.data_ptr() == tc.data_ptr()
    assert torch.equal(a.dlogits.view(torch.int16 if bf16 else torch.int32),
                       b.dlogits.view(torch.int16 if bf16 else torch.int32))
    assert torch.equal(a.loss, b.loss) and torch.equal(a.lse, b.lse)
