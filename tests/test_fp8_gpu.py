"""GPU parity of the FP8 operand variant against the float64 oracle: the
oracle's logits come from the dequantised E4M3 operands (scale x e4m3), its
gradient products from the bf16 tensors the operands were quantised from."""
import numpy as np
import pytest

import flce_inputs
import oracle
from flce_testlib import assert_within, compare, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import linear_cross_entropy_flce_gb300 as flce


def _case(wl):
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H8, sh = flce_inputs.to_fp8_per_tensor(Hb)
    W8, sw = flce_inputs.to_fp8_per_tensor(Wb)
    dev = torch.device("cuda:0")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    H, W, lab = to_device(Hb, Wb, y)
    He = flce_inputs.e4m3_decode(H8) * np.float64(sh)
    We = flce_inputs.e4m3_decode(W8) * np.float64(sw)
    return (t(H8), float(sh), t(W8), float(sw), lab, H, W), (He, We, Hb, Wb, y)


@pytest.mark.parametrize("shape", [(300, 256, 3000), (129, 144, 1500), (64, 128, 1000)])
def test_fp8_forward_backward_parity(shape):
    N, D, V = shape
    wl = flce_inputs.Workload("fp8", N, D, V, 1.0, 0.05, "uniform", 0.07, seed=N + D)
    (H8, sh, W8, sw, lab, H, W), (He, We, Hb, Wb, y) = _case(wl)
    res = flce.forward_backward_fp8(H8, sh, W8, sw, lab, H, W)
    assert flce.check_status(res.status) == flce.FLCE_OK
    ref = oracle.flce(He, We, y, Hg=flce_inputs.bf16_bits_to_f64(Hb),
                      Wg=flce_inputs.bf16_bits_to_f64(Wb))
    errs = compare(res, ref)
    print(errs)
    assert_within(errs)


def test_fp8_forward_only_and_llama2_workload():
    (H8, sh, W8, sw, lab, H, W), (He, We, Hb, Wb, y) = _case(flce_inputs.get("llama2"))
    fwd = flce.forward_backward_fp8(H8, sh, W8, sw, lab, need_dh=False, need_dw=False)
    full = flce.forward_backward_fp8(H8, sh, W8, sw, lab, H, W)
    assert flce.check_status(full.status) == flce.FLCE_OK
    torch.cuda.synchronize()
    assert torch.equal(fwd.loss, full.loss) and torch.equal(fwd.lse, full.lse)
    ref = oracle.flce(He, We, y, Hg=flce_inputs.bf16_bits_to_f32(Hb),
                      Wg=flce_inputs.bf16_bits_to_f32(Wb))
    errs = compare(full, ref)
    print(errs)
    assert_within(errs)


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
                      Wg=flce_inputs.bf16_bits_to_f64(Wb))
    errs = compare(res, ref)
    print(errs)
    assert_within(errs)
