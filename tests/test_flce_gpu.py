"""GPU parity of the CUDA path (through the C ABI) against the CPU float64
oracle on the same seeded inputs, plus edge cases and invariants that hold at
any size."""
import numpy as np
import pytest

import flce_inputs
import oracle
from flce_testlib import (assert_within, bf16_tensor_to_f64, compare, dw_sample_groups, oracle_check,
                          tensor_to_f64, to_device)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import linear_cross_entropy_flce_gb300 as flce


def _inputs(N, D, V, seed=0, w_std=0.05, h_scale=1.0, p_ignore=0.0, labels="uniform"):
    wl = flce_inputs.Workload("custom", N, D, V, h_scale, w_std, labels, p_ignore, seed=seed)
    return flce_inputs.make_inputs(wl)


def _run_and_compare(Hb, Wb, y, **opts):
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab, **opts)
    assert flce.check_status(res.status) == flce.FLCE_OK
    ref_kw = {k: opts[k] for k in ("reduction", "grad_scale", "normalizer", "ignore_index") if k in opts}
    ref = oracle.flce(flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb), y,
                      want_abs=True, **ref_kw)
    oracle_check(res, Hb, Wb, y, ref, opts)
    return res, ref


def test_tiny_workload_full_parity():
    Hb, Wb, y = flce_inputs.make_inputs(flce_inputs.get("tiny"))
    _run_and_compare(Hb, Wb, y)


@pytest.mark.parametrize("opts", [
    {},
    {"v_chunk": 512, "n_block": 128},
    {"v_chunk": 256, "n_block": 256, "v_splits": 3},
    {"v_chunk": 768, "n_block": 128, "dw_dtype": "bfloat16"},
    {"dw_dtype": "bfloat16"},
])
def test_ragged_shapes_and_plans(opts):
    # N, V not multiples of the 128 x 256 tile; D not a multiple of 64.
    Hb, Wb, y = _inputs(300, 200, 1500, seed=3, p_ignore=0.07)
    _run_and_compare(Hb, Wb, y, **opts)


@pytest.mark.parametrize("N,D,V", [(1, 8, 1), (1, 64, 2), (129, 136, 257), (127, 8, 300), (512, 1024, 4096)])
def test_small_and_degenerate_shapes(N, D, V):
    Hb, Wb, y = _inputs(N, D, V, seed=N + V)
    _run_and_compare(Hb, Wb, y)


@pytest.mark.parametrize("N,D,V,opts", [
    (300, 576, 1500, {}),                          # second 256-wide half of tile 1 wholly past D
    (257, 704, 2049, {"v_chunk": 1024}),           # half 0 of tile 1 ragged, half 1 past D
    (520, 1088, 3000, {"n_block": 256, "dw_dtype": "bfloat16"}),  # 2 tiles + 64 columns, bf16 dW over token blocks
    (130, 840, 700, {}),                           # D % 64 != 0: two-box MN-major loads, halves past D
])
def test_wide_dw_tile_edges(N, D, V, opts):
    """The dW product's 256 x 512 tiles where D is not a multiple of 512: a tile's
    second N = 256 half lies partly or wholly past D (its B rows read the zero fill
    of the copy engine, its output columns are clipped by the store map)."""
    Hb, Wb, y = _inputs(N, D, V, seed=N + D + V, p_ignore=0.05)
    _run_and_compare(Hb, Wb, y, **opts)


@pytest.mark.parametrize("N,D,V", [(200, 16384, 3000), (300, 8200, 2000)])
def test_large_hidden_sizes(N, D, V):
    """Hidden sizes of the largest heads: D = 16384 (256 K blocks in the logits
    products, 32 wide dW tiles across D), and D = 8200, not a multiple of 64 (the
    MN-major H and W operands of dW and dH then load as two 2-D boxes per half)."""
    Hb, Wb, y = _inputs(N, D, V, seed=D, w_std=0.01, p_ignore=0.05)
    _run_and_compare(Hb, Wb, y)


def test_one_label_for_every_token():
    """Every valid token has the same label: dW row y sums 1900 one-hot terms of
    -scale h_i, so its softmax part is about 1e-4 of the row and only the fp32
    accumulation allowance of the gate separates rounding from error there; every
    other row is all softmax part."""
    Hb, Wb, y = _inputs(2000, 256, 3000, seed=26, p_ignore=0.05)
    y[y != -100] = 7
    _run_and_compare(Hb, Wb, y)


@pytest.mark.parametrize("opts", [{}, {"v_splits": 3}])
def test_peaked_logits_online_lse(opts):
    """Logits with a standard deviation of about 30 (the online maximum jumps by
    tens between vocabulary tiles, and each row's softmax is close to one-hot),
    half of the labels on the row's largest logit (p close to 1, so the target
    entry of G is a difference of nearly equal numbers) and half uniform (p close
    to 0)."""
    Hb, Wb, y = _inputs(300, 256, 3000, seed=31, w_std=0.5, h_scale=4.0, p_ignore=0.05)
    Z = flce_inputs.bf16_bits_to_f64(Hb) @ flce_inputs.bf16_bits_to_f64(Wb).T
    assert Z.std() > 20.0
    top = np.argmax(Z, axis=1).astype(np.int32)
    half = np.arange(len(y)) % 2 == 0
    y = np.where((y != -100) & half, top, y).astype(np.int32)
    _run_and_compare(Hb, Wb, y, **opts)


def test_targets_far_below_a_flat_maximum():
    """Most logits of a row equal (the maximum shared by about 2950 ids) and the
    target 70-86 below it: the target's term is a normal fp32 number far smaller
    than the sum of the others, whose ratio to it would overflow fp32 (the loss
    must stay finite and equal the oracle's)."""
    N, D, V = 128, 64, 3000
    H = np.zeros((N, D), dtype=np.float32)
    H[:, 0] = 10.0
    H[:, 1] = np.linspace(-1.0, 1.0, N, dtype=np.float32)
    W = np.zeros((V, D), dtype=np.float32)
    W[:, 0] = 1.0
    targets = np.arange(50)
    W[targets, 0] = -7.5 + 0.02 * targets.astype(np.float32)   # z about -75 .. -65
    y = (np.arange(N) % 50).astype(np.int32)
    y[::17] = -100
    Hb, Wb = flce_inputs.f32_to_bf16_bits(H), flce_inputs.f32_to_bf16_bits(W)
    res, ref = _run_and_compare(Hb, Wb, y)
    assert np.isfinite(float(res.loss.item())) and ref["loss"] > 70.0


def test_labels_at_vocabulary_edges():
    Hb, Wb, y = _inputs(256, 128, 1000, seed=5)
    y[:64] = 0
    y[64:128] = 999
    _run_and_compare(Hb, Wb, y)


@pytest.mark.parametrize("opts", [
    {"reduction": "sum"},
    {"grad_scale": 0.25},
    {"grad_scale": -1.5},   # a negative upstream factor flips every gradient's sign
    {"normalizer": 1000.0},
    {"ignore_index": 7},
])
def test_reduction_and_scaling_options(opts):
    Hb, Wb, y = _inputs(200, 256, 700, seed=9, p_ignore=0.1)
    if opts.get("ignore_index") == 7:
        y[y == -100] = 7
    _run_and_compare(Hb, Wb, y, **opts)


def test_all_tokens_ignored():
    Hb, Wb, y = _inputs(130, 64, 400, seed=11)
    y[:] = -100
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab, v_chunk=256)
    assert flce.check_status(res.status) == flce.FLCE_OK
    assert float(res.loss.item()) == 0.0
    assert torch.count_nonzero(res.dH).item() == 0
    assert torch.count_nonzero(res.dW).item() == 0
    ref = oracle.flce(flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb), y)
    assert np.max(np.abs(res.lse.double().cpu().numpy() - ref["lse"])) <= 2e-3


def test_zero_weights_closed_form():
    """W = 0: loss and every lse equal log V, dH = 0, dW_v = sum_valid (1/V - [y=v]) h_i / n."""
    N, D, V = 300, 128, 1000
    Hb, _, y = _inputs(N, D, V, seed=12, p_ignore=0.1)
    Wb = np.zeros((V, D), dtype=np.uint16)
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab, v_chunk=256)
    assert flce.check_status(res.status) == flce.FLCE_OK
    assert float(res.loss.item()) == pytest.approx(np.log(V), rel=1e-6)
    assert np.max(np.abs(res.lse.cpu().numpy() - np.log(V))) < 1e-5
    assert torch.count_nonzero(res.dH).item() == 0
    Hd = flce_inputs.bf16_bits_to_f64(Hb)
    valid = y != -100
    n = valid.sum()
    expect = np.tile(Hd[valid].sum(0) / V / n, (V, 1))
    for i in np.nonzero(valid)[0]:
        expect[y[i]] -= Hd[i] / n
    got = res.dW.double().cpu().numpy()
    assert np.linalg.norm(got - expect) / np.linalg.norm(expect) < 5e-3


def test_ignored_rows_have_exactly_zero_dh():
    Hb, Wb, y = _inputs(400, 256, 2000, seed=13, p_ignore=0.2)
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab)
    ign = torch.from_numpy(y == -100).to(res.dH.device)
    assert torch.count_nonzero(res.dH[ign]).item() == 0


def test_dw_columns_sum_to_zero():
    """sum_v dW_v = sum_i (sum_v g_iv) h_i = 0 (rows of softmax - onehot sum to 0)."""
    Hb, Wb, y = _inputs(512, 256, 3000, seed=14)
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab)
    colsum = res.dW.double().sum(0)
    scale = res.dW.double().abs().sum(0)
    assert float((colsum.abs() / scale).max()) < 5e-3


def test_several_tiles_per_pair_and_partial_last_k_stage():
    """dW and dH launches with more tiles than the 76 cluster pairs, so that pairs run
    tiles in both K directions, and K extents (2460 tokens; a 9760-id last chunk) that
    leave the last ring stage half filled."""
    Hb, Wb, y = _inputs(2460, 2048, 20000, seed=21, p_ignore=0.05)
    _run_and_compare(Hb, Wb, y, v_chunk=10240)


def test_run_to_run_bitwise_determinism():
    Hb, Wb, y = _inputs(700, 512, 5000, seed=15, p_ignore=0.05)
    H, W, lab = to_device(Hb, Wb, y)
    a = flce.forward_backward(H, W, lab, v_chunk=1024, n_block=256)
    b = flce.forward_backward(H, W, lab, v_chunk=1024, n_block=256)
    torch.cuda.synchronize()
    assert torch.equal(a.loss, b.loss) and torch.equal(a.lse, b.lse)
    assert torch.equal(a.dH.view(torch.int16), b.dH.view(torch.int16))
    assert torch.equal(a.dW, b.dW)


def test_full_size_bitwise_determinism():
    """The long-sequence head (32768 tokens: 4 token blocks x 8 vocabulary chunks,
    so dW is reduce-added across blocks and dH across chunks, each in launch
    order, by the merged dH + dW launches of 760 units on every SM) gives the same
    bits twice; the second call runs in a workspace left dirty by the first."""
    wl = flce_inputs.get("long_seq")
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    del Hb, Wb
    ws = torch.empty(flce.workspace_size(wl.N, wl.D, wl.V), dtype=torch.uint8, device=H.device)
    a = flce.forward_backward(H, W, lab, workspace=ws)
    b = flce.forward_backward(H, W, lab, workspace=ws)
    torch.cuda.synchronize()
    assert flce.check_status(a.status) == flce.FLCE_OK and flce.check_status(b.status) == flce.FLCE_OK
    assert torch.equal(a.loss, b.loss) and torch.equal(a.lse, b.lse)
    assert torch.equal(a.dH.view(torch.int16), b.dH.view(torch.int16))
    assert torch.equal(a.dW.view(torch.int32), b.dW.view(torch.int32))


def test_optional_outputs_and_forward_only():
    Hb, Wb, y = _inputs(300, 128, 900, seed=16, p_ignore=0.1)
    H, W, lab = to_device(Hb, Wb, y)
    full = flce.forward_backward(H, W, lab)
    only_dh = flce.forward_backward(H, W, lab, need_dw=False)
    only_dw = flce.forward_backward(H, W, lab, need_dh=False)
    fwd = flce.forward(H, W, lab)
    torch.cuda.synchronize()
    assert torch.equal(full.dH.view(torch.int16), only_dh.dH.view(torch.int16))
    assert torch.equal(full.dW, only_dw.dW)
    assert torch.equal(full.loss, fwd.loss) and torch.equal(full.lse, fwd.lse)


def test_label_out_of_range_sets_device_status():
    Hb, Wb, y = _inputs(200, 64, 500, seed=17)
    y[33] = 500
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab)
    assert flce.check_status(res.status) == flce.FLCE_ERR_LABEL_RANGE
    y[33] = -3
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab)
    assert flce.check_status(res.status) == flce.FLCE_ERR_LABEL_RANGE


def test_workspace_too_small_is_rejected():
    Hb, Wb, y = _inputs(200, 64, 500, seed=18)
    H, W, lab = to_device(Hb, Wb, y)
    need = flce.workspace_size(200, 64, 500)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda:0")
    with pytest.raises(flce.FLCEError) as e:
        flce.forward_backward(H, W, lab, workspace=ws)
    assert e.value.code == flce.FLCE_ERR_WORKSPACE


def test_token_permutation_equivariance():
    """Each token's logits row, lse and dH row depend only on that token, so
    permuting whole 128-token blocks of rows permutes lse and dH bit for bit."""
    Hb, Wb, y = _inputs(512, 256, 2000, seed=19, p_ignore=0.05)
    perm = np.concatenate([np.arange(256, 384), np.arange(0, 128), np.arange(384, 512),
                           np.arange(128, 256)])
    a = flce.forward_backward(*to_device(Hb, Wb, y), v_splits=2)
    b = flce.forward_backward(*to_device(Hb[perm], Wb, y[perm]), v_splits=2)
    torch.cuda.synchronize()
    pt = torch.from_numpy(perm).to(a.lse.device)
    assert torch.equal(a.lse[pt], b.lse)
    assert torch.equal(a.dH[pt].view(torch.int16), b.dH.view(torch.int16))
    assert abs(float(a.loss.item()) - float(b.loss.item())) <= 1e-6 * abs(float(a.loss.item()))


def test_llama2_like_workload_full_parity():
    Hb, Wb, y = flce_inputs.make_inputs(flce_inputs.get("llama2"))
    _run_and_compare(Hb, Wb, y)


@pytest.mark.parametrize("name", ["llama3_8b", "qwen2_7b", "long_seq"])
def test_full_size_workload_sampled_parity(name):
    """Full-size workloads in the default plan (the launch configuration the
    benchmark times): loss and every token's lse against the oracle, dH on 256
    sampled tokens and dW on 64 sampled vocabulary ids, the ids gated in three
    groups (frequent labels, uniform picks, V-1) and the softmax part of both
    gradients gated on its own."""
    wl = flce_inputs.get(name)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab)
    assert flce.check_status(res.status) == flce.FLCE_OK
    del H, W
    rows = oracle.sample_rows(y, 256, seed=wl.seed)
    vids = oracle.sample_vocab(y, wl.V, 64, seed=wl.seed)
    Hf, Wf = flce_inputs.bf16_bits_to_f32(Hb), flce_inputs.bf16_bits_to_f32(Wb)
    ref = oracle.flce(Hf, Wf, y, dh_rows=rows, dw_rows=vids, want_abs=True)
    dev = res.lse.device
    groups = dw_sample_groups(y, vids, wl.V)
    assert set(groups) >= {"last", "frequent", "uniform"}
    errs = compare(res, ref, dh_rows=torch.from_numpy(rows).to(dev),
                   dw_rows=torch.from_numpy(vids).to(dev), labels=y, Hg=Hf, Wg=Wf,
                   dw_groups=groups)
    print(name, errs)
    assert_within(errs)
    # no [N, V] buffer: the whole extra device memory is the declared workspace
    assert flce.workspace_size(wl.N, wl.D, wl.V) < wl.N * wl.V * 4 // 8
    if name == "long_seq":
        # bf16 dW over the plan's four token blocks: the fp32 dW accumulator in the
        # workspace, added to in launch order, rounded once at the end
        del res
        H, W, lab = to_device(Hb, Wb, y)
        r16 = flce.forward_backward(H, W, lab, dw_dtype="bfloat16")
        assert flce.check_status(r16.status) == flce.FLCE_OK
        assert flce.get_plan(wl.N, wl.D, wl.V)["n_blocks"] > 1
        del H, W
        errs16 = compare(r16, ref, dh_rows=torch.from_numpy(rows).to(dev),
                         dw_rows=torch.from_numpy(vids).to(dev), labels=y, Hg=Hf, Wg=Wf,
                         opts={"dw_dtype": "bfloat16"}, dw_groups=groups)
        print(name, "bf16 dW", errs16)
        assert_within(errs16)


def test_bounded_wait_timeout_sets_status_and_context_stays_usable():
    """A 1-ns limit makes the kernels' pipeline waits run out: the call must end
    (no hang), report FLCE_ERR_TIMEOUT through the status word, and leave the
    CUDA context usable, so that the next normal call is correct."""
    Hb, Wb, y = _inputs(128, 64, 256, seed=23)
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab, timeout_ns=1)
    assert flce.check_status(res.status) == flce.FLCE_ERR_TIMEOUT
    _run_and_compare(Hb, Wb, y)


def test_forward_per_token_loss_reduction_none():
    """reduction="none" (forward only): each token's lse_i - z_{i,y_i}, 0 for
    ignored tokens, against the oracle's per-token NLL; the backward rejects it."""
    Hb, Wb, y = _inputs(333, 256, 3000, seed=24, p_ignore=0.1)
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward(H, W, lab, reduction="none")
    assert flce.check_status(res.status) == flce.FLCE_OK
    ref = oracle.flce(flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb), y,
                      want_grads=False)
    per = res.loss.double().cpu().numpy()
    assert per.shape == (333,)
    assert np.max(np.abs(per - ref["nll"])) <= 2e-3
    assert np.all(per[y == -100] == 0.0)
    mean = flce.forward(H, W, lab)
    assert abs(per[y != -100].mean() - float(mean.loss.item())) <= 1e-5 * float(mean.loss.item())
    with pytest.raises(flce.FLCEError) as e:
        flce.forward_backward(H, W, lab, reduction="none")
    assert e.value.code == flce.FLCE_ERR_OPTION


def test_forward_only_matches_oracle_on_llama2_workload():
    """The evaluation path alone (flce_forward) on the Llama-2-like head."""
    Hb, Wb, y = flce_inputs.make_inputs(flce_inputs.get("llama2"))
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward(H, W, lab)
    assert flce.check_status(res.status) == flce.FLCE_OK
    ref = oracle.flce(flce_inputs.bf16_bits_to_f32(Hb), flce_inputs.bf16_bits_to_f32(Wb), y,
                      want_grads=False)
    assert abs(float(res.loss.item()) - ref["loss"]) <= 1e-3 * ref["loss"]
    assert np.max(np.abs(res.lse.double().cpu().numpy() - ref["lse"])) <= 2e-3


def test_million_token_vocabulary_full_parity():
    """V >= 1M (the open question on the lecture page about very large
    vocabularies): 1,100,000 ids, a ragged final tile, 68 vocabulary chunks in
    the default plan; every lse, dH and dW element against the oracle."""
    N, D, V = 300, 128, 1_100_000
    Hb, Wb, y = _inputs(N, D, V, seed=25, w_std=0.05, p_ignore=0.05)
    H, W, lab = to_device(Hb, Wb, y)
    res = flce.forward_backward(H, W, lab)
    assert flce.check_status(res.status) == flce.FLCE_OK
    plan = flce.get_plan(N, D, V)
    assert plan["n_chunks"] > 8
    ref = oracle.flce(flce_inputs.bf16_bits_to_f32(Hb), flce_inputs.bf16_bits_to_f32(Wb), y,
                      row_block=32, want_abs=True)
    oracle_check(res, Hb, Wb, y, ref)
