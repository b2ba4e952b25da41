"""GPU parity of the FP8 operand variant against the float64 oracle: the
oracle's logits come from the dequantised E4M3 operands (scale x e4m3), its
gradient products from the bf16 tensors the operands were quantised from."""
import numpy as np
import pytest

import flce_inputs
import oracle
from oracle import e4m3
from flce_testlib import assert_within, compare, dw_sample_groups, oracle_check, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import linear_cross_entropy_flce_gb300 as flce


def _case(wl):
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    qh = e4m3.quantize_per_tensor(flce_inputs.bf16_bits_to_f32(Hb))
    qw = e4m3.quantize_per_tensor(flce_inputs.bf16_bits_to_f32(Wb))
    H8, sh, W8, sw = qh["codes"], qh["scale"], qw["codes"], qw["scale"]
    dev = torch.device("cuda:0")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    H, W, lab = to_device(Hb, Wb, y)
    He = e4m3.e4m3_decode(H8) * np.float64(sh)
    We = e4m3.e4m3_decode(W8) * np.float64(sw)
    return (t(H8), float(sh), t(W8), float(sw), lab, H, W), (He, We, Hb, Wb, y)


@pytest.mark.parametrize("shape", [(300, 256, 3000), (129, 144, 1500), (64, 128, 1000)])
def test_fp8_forward_backward_parity(shape):
    N, D, V = shape
    wl = flce_inputs.Workload("fp8", N, D, V, 1.0, 0.05, "uniform", 0.07, seed=N + D)
    (H8, sh, W8, sw, lab, H, W), (He, We, Hb, Wb, y) = _case(wl)
    res = flce.forward_backward_fp8(H8, sh, W8, sw, lab, H, W)
    assert flce.check_status(res.status) == flce.FLCE_OK
    ref = oracle.flce(He, We, y, Hg=flce_inputs.bf16_bits_to_f64(Hb),
                      Wg=flce_inputs.bf16_bits_to_f64(Wb), want_abs=True)
    oracle_check(res, Hb, Wb, y, ref)


def test_fp8_forward_only_and_llama2_workload():
    (H8, sh, W8, sw, lab, H, W), (He, We, Hb, Wb, y) = _case(flce_inputs.get("llama2"))
    fwd = flce.forward_backward_fp8(H8, sh, W8, sw, lab, need_dh=False, need_dw=False)
    full = flce.forward_backward_fp8(H8, sh, W8, sw, lab, H, W)
    assert flce.check_status(full.status) == flce.FLCE_OK
    torch.cuda.synchronize()
    assert torch.equal(fwd.loss, full.loss) and torch.equal(fwd.lse, full.lse)
    ref = oracle.flce(He, We, y, Hg=flce_inputs.bf16_bits_to_f32(Hb),
                      Wg=flce_inputs.bf16_bits_to_f32(Wb), want_abs=True)
    oracle_check(full, Hb, Wb, y, ref)


@pytest.mark.parametrize("opts", [{"v_chunk": 512, "n_block": 256},
                                  {"v_chunk": 768, "n_block": 128, "dw_dtype": "bfloat16"}])
def test_fp8_token_blocks_and_chunks(opts):
    """The FP8 variant under plans with several vocabulary chunks and token
    blocks (dH accumulated over chunks, dW over token blocks, bf16 dW)."""
    wl = flce_inputs.Workload("fp8plan", 300, 200 + 56, 1500, 1.0, 0.05, "uniform", 0.07, seed=5)
    (H8, sh, W8, sw, lab, H, W), (He, We, Hb, Wb, y) = _case(wl)
    res = flce.forward_backward_fp8(H8, sh, W8, sw, lab, H, W, **opts)
    assert flce.check_status(res.status) == flce.FLCE_OK
    ref = oracle.flce(He, We, y, Hg=flce_inputs.bf16_bits_to_f64(Hb),
                      Wg=flce_inputs.bf16_bits_to_f64(Wb), want_abs=True)
    oracle_check(res, Hb, Wb, y, ref, opts)


def _wide_range_bf16(shape, seed):
    """bf16 bits spanning E4M3's whole range after scaling: N(0,1) times 10^u,
    u uniform in [-7, 1], so codes land in the subnormals, the normals and at 448."""
    g = np.random.default_rng(seed)
    x = g.standard_normal(shape).astype(np.float32) * np.float32(10.0) ** g.uniform(-7, 1, shape).astype(np.float32)
    return flce_inputs.f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("case", ["normal", "wide", "zeros", "tiny", "ragged_grid", "subnormal"])
def test_device_quantizer_matches_its_definition(case):
    """flce_quantize_e4m3 bit for bit against the oracle's per-tensor E4M3
    quantisation (oracle/e4m3.py, pinned by its properties on the CPU)."""
    if case == "normal":
        bits = flce_inputs.normal_bf16((300, 256), 0.05, seed=3, stream=0)
    elif case == "wide":
        bits = _wide_range_bf16((517, 96), seed=4)
    elif case == "zeros":
        bits = np.zeros((16, 64), dtype=np.uint16)
        bits[3, 5] = 0x8000  # -0 counts as zero
    elif case == "tiny":
        bits = flce_inputs.normal_bf16((1, 8), 1.0, seed=5, stream=0)
    elif case == "subnormal":  # amax ~1e-39: 448 / amax overflows fp32, inv is capped
        x = np.random.default_rng(7).uniform(-1, 1, (64, 40)).astype(np.float32) * np.float32(1e-39)
        bits = flce_inputs.f32_to_bf16_bits(x)
    else:  # more 8-element groups than one grid pass covers
        bits = _wide_range_bf16((4099, 2056), seed=6)
    r = e4m3.quantize_per_tensor(flce_inputs.bf16_bits_to_f32(bits))
    q_ref, scale_ref, amax_ref = r["codes"], r["scale"], r["amax"]
    x = torch.from_numpy(bits.view(np.int16)).to("cuda:0").view(torch.bfloat16)
    q, out = flce.quantize_e4m3(x)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert o[1] == amax_ref and o[0] == scale_ref, (o, amax_ref, scale_ref)
    qd = q.cpu().numpy()
    bad = np.flatnonzero(qd.ravel() != q_ref.ravel())
    assert bad.size == 0, (bad[:8], qd.ravel()[bad[:8]], q_ref.ravel()[bad[:8]])


def test_device_quantized_operands_feed_the_fp8_path():
    """H8, W8 and their scales made on the device (scales passed as device scalars,
    no host round trip) give the oracle's result over the dequantised operands."""
    wl = flce_inputs.Workload("fp8q", 300, 256, 3000, 1.0, 0.05, "uniform", 0.07, seed=11)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    H8, oh = flce.quantize_e4m3(H)
    W8, ow = flce.quantize_e4m3(W)
    res = flce.forward_backward_fp8(H8, oh[0:1], W8, ow[0:1], lab, H, W)
    assert flce.check_status(res.status) == flce.FLCE_OK
    torch.cuda.synchronize()
    He = e4m3.e4m3_decode(H8.cpu().numpy()) * np.float64(oh[0].item())
    We = e4m3.e4m3_decode(W8.cpu().numpy()) * np.float64(ow[0].item())
    ref = oracle.flce(He, We, y, Hg=flce_inputs.bf16_bits_to_f64(Hb),
                      Wg=flce_inputs.bf16_bits_to_f64(Wb), want_abs=True)
    oracle_check(res, Hb, Wb, y, ref)


def test_fp8_full_size_llama3_workload_sampled_parity():
    """The FP8 variant at the Llama-3-8B-shaped head in the launch configuration the
    benchmark times (operands quantised on the device, scales read from device
    memory): loss and every lse against the oracle over the dequantised operands,
    dH on 256 sampled tokens and dW on 64 sampled ids in their three groups, the
    softmax part and the element-wise bound included."""
    wl = flce_inputs.get("llama3_8b")
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    H8, oh = flce.quantize_e4m3(H)
    W8, ow = flce.quantize_e4m3(W)
    res = flce.forward_backward_fp8(H8, oh[0:1], W8, ow[0:1], lab, H, W)
    assert flce.check_status(res.status) == flce.FLCE_OK
    He = (e4m3.e4m3_decode(H8.cpu().numpy()) * np.float64(oh[0].item())).astype(np.float32)
    We = (e4m3.e4m3_decode(W8.cpu().numpy()) * np.float64(ow[0].item())).astype(np.float32)
    del H, W, H8, W8
    rows = oracle.sample_rows(y, 256, seed=wl.seed)
    vids = oracle.sample_vocab(y, wl.V, 64, seed=wl.seed)
    Hf, Wf = flce_inputs.bf16_bits_to_f32(Hb), flce_inputs.bf16_bits_to_f32(Wb)
    ref = oracle.flce(He, We, y, Hg=Hf, Wg=Wf, dh_rows=rows, dw_rows=vids, want_abs=True)
    dev = res.lse.device
    errs = compare(res, ref, dh_rows=torch.from_numpy(rows).to(dev),
                   dw_rows=torch.from_numpy(vids).to(dev), labels=y, Hg=Hf, Wg=Wf,
                   dw_groups=dw_sample_groups(y, vids, wl.V))
    print(errs)
    assert_within(errs)
