"""The drop-in loss under PyTorch autograd: loss.backward() must fill the
parameters' gradients with the oracle's dH and dW, scaled by the upstream
gradient, and run the forward alone when no gradient is needed."""
import numpy as np
import pytest

import flce_inputs
import oracle
from flce_testlib import rel_fro, tensor_to_f64, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import linear_cross_entropy_flce_gb300 as flce


def _case(N=300, D=256, V=3000, seed=51, p_ignore=0.1):
    wl = flce_inputs.Workload("autograd", N, D, V, 1.0, 0.05, "uniform", p_ignore, seed=seed)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    ref = oracle.flce(flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb), y)
    return Hb, Wb, y, ref


def test_backward_matches_oracle():
    Hb, Wb, y, ref = _case()
    H, W, lab = to_device(Hb, Wb, y)
    H.requires_grad_(True)
    W.requires_grad_(True)
    loss = flce.FusedLinearCrossEntropyLoss()(H, W, lab.to(torch.int64))
    assert loss.dim() == 0
    loss.backward()
    assert abs(float(loss.item()) - ref["loss"]) <= 1e-3 * ref["loss"]
    assert H.grad.dtype == torch.bfloat16 and W.grad.dtype == torch.bfloat16
    assert rel_fro(tensor_to_f64(H.grad), ref["dH"]) <= 5e-3
    assert rel_fro(tensor_to_f64(W.grad), ref["dW"]) <= 5e-3


def test_upstream_gradient_scales_and_batched_shapes():
    Hb, Wb, y, ref = _case(N=256, seed=52)
    H, W, lab = to_device(Hb, Wb, y)
    H3 = H.reshape(2, 128, -1).detach().requires_grad_(True)
    W.requires_grad_(True)
    loss = flce.fused_linear_cross_entropy(H3, W, lab.reshape(2, 128))
    (loss * 3.0).backward()
    assert H3.grad.shape == H3.shape
    assert rel_fro(tensor_to_f64(H3.grad.reshape(256, -1)), 3.0 * ref["dH"]) <= 5e-3
    assert rel_fro(tensor_to_f64(W.grad), 3.0 * ref["dW"]) <= 5e-3


def test_only_the_requested_gradients_and_no_grad_forward():
    Hb, Wb, y, ref = _case(seed=53)
    H, W, lab = to_device(Hb, Wb, y)
    W.requires_grad_(True)
    loss = flce.FusedLinearCrossEntropyLoss(reduction="sum")(H, W, lab)
    loss.backward()
    assert H.grad is None
    assert rel_fro(tensor_to_f64(W.grad), ref["dW"] * ref["n_valid"]) <= 5e-3
    with torch.no_grad():
        l2 = flce.FusedLinearCrossEntropyLoss()(H, W, lab)
    assert abs(float(l2.item()) - ref["loss"]) <= 1e-3 * ref["loss"]
    per = flce.FusedLinearCrossEntropyLoss(reduction="none")(H, W.detach(), lab)
    assert per.shape == lab.shape
    assert np.max(np.abs(per.double().cpu().numpy() - ref["nll"])) <= 2e-3
