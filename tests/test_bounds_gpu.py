"""Writes stay inside their buffers, and invariants of the method that need no
oracle hold on the GPU path.

- Canaries: every output and the workspace sit inside larger allocations whose
  guard bytes carry a pattern; ragged shapes and several plans (vocabulary chunks,
  token blocks, bf16 dW accumulated over token blocks, a single chunk that writes
  bf16 dH directly) must leave every guard byte untouched (the copy engine clips
  ragged output tiles at the map edges).
- Shift invariance: adding the same vector c to every row of W adds h_i . c to
  every logit of token i, so lse shifts by h_i . c while the loss, G, dH and dW do
  not change. W and c are multiples of 2^-10 small enough that W + c is exact in
  bf16, so the shifted problem is the same problem."""
import numpy as np
import pytest

import flce_inputs
import oracle
from flce_testlib import oracle_check, rel_fro, tensor_to_f64, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import linear_cross_entropy_flce_gb300 as flce

GUARD = 4096  # bytes on each side
PATTERN = 0xA5


def _guarded(nbytes, dev):
    buf = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=dev)
    return buf, buf[GUARD:GUARD + nbytes]


def _guards_intact(buf):
    host = buf.cpu().numpy()
    return bool((host[:GUARD] == PATTERN).all() and (host[-GUARD:] == PATTERN).all())


@pytest.mark.parametrize("N,D,V,opts", [
    (300, 200, 1500, {"v_chunk": 512, "n_block": 256}),
    (300, 200, 1500, {"v_chunk": 768, "n_block": 128, "dw_dtype": "bfloat16"}),
    (257, 136, 1000, {}),                       # one chunk: dH written as bf16 directly
    (513, 264, 4097, {"v_chunk": 1024}),
])
def test_outputs_and_workspace_stay_inside_their_buffers(N, D, V, opts):
    wl = flce_inputs.Workload("guard", N, D, V, 1.0, 0.05, "uniform", 0.05, seed=N + D)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    dev = H.device
    dw_bf16 = opts.get("dw_dtype") == "bfloat16"
    bufs = {}
    bufs["loss"], loss = _guarded(4, dev)
    bufs["lse"], lse = _guarded(N * 4, dev)
    bufs["dH"], dh = _guarded(N * D * 2, dev)
    bufs["dW"], dw = _guarded(V * D * (2 if dw_bf16 else 4), dev)
    ws_bytes = flce.workspace_size(N, D, V, flce.make_options(**opts))
    bufs["ws"], ws = _guarded(ws_bytes, dev)
    out = {"loss": loss.view(torch.float32), "lse": lse.view(torch.float32),
           "dH": dh.view(torch.bfloat16).view(N, D),
           "dW": dw.view(torch.bfloat16 if dw_bf16 else torch.float32).view(V, D)}
    res = flce.forward_backward(H, W, lab, out=out, workspace=ws, **opts)
    assert flce.check_status(res.status) == flce.FLCE_OK
    for k, b in bufs.items():
        assert _guards_intact(b), k
    ref = oracle.flce(flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb), y,
                      want_abs=True)
    oracle_check(res, Hb, Wb, y, ref, opts)


def test_shift_of_every_weight_row_changes_only_lse():
    N, D, V = 384, 256, 2000
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([7, 77])))
    # multiples of 2^-10 with |k| <= 100 for W and |k| <= 60 for c: W + c has
    # |k| <= 160 < 256, so every element is exact in bf16
    Wq = g.integers(-100, 101, size=(V, D)).astype(np.float32) / 1024.0
    c = g.integers(-60, 61, size=D).astype(np.float32) / 1024.0
    Hb = flce_inputs.normal_bf16((N, D), 0.5, 7, 1)
    y = g.integers(0, V, size=N).astype(np.int32)
    y[:20] = -100
    Wb = flce_inputs.f32_to_bf16_bits(Wq)
    Wsb = flce_inputs.f32_to_bf16_bits(Wq + c[None, :])
    assert np.array_equal(flce_inputs.bf16_bits_to_f32(Wsb), Wq + c[None, :])
    H, W, lab = to_device(Hb, Wb, y)
    _, Ws, _ = to_device(Hb, Wsb, y)
    a = flce.forward_backward(H, W, lab)
    b = flce.forward_backward(H, Ws, lab)
    assert flce.check_status(a.status) == flce.FLCE_OK and flce.check_status(b.status) == flce.FLCE_OK
    la, lb = float(a.loss.item()), float(b.loss.item())
    assert abs(la - lb) <= 1e-5 * abs(la)
    hc = flce_inputs.bf16_bits_to_f64(Hb) @ c.astype(np.float64)
    dl = b.lse.double().cpu().numpy() - a.lse.double().cpu().numpy()
    assert np.max(np.abs(dl - hc)) <= 2e-3
    assert rel_fro(tensor_to_f64(b.dH), tensor_to_f64(a.dH)) <= 5e-3
    assert rel_fro(tensor_to_f64(b.dW), tensor_to_f64(a.dW)) <= 5e-3


@pytest.mark.parametrize("N,V,bf16", [(40, 128256, False), (24, 128257, True), (4, 240007, False),
                                      (33, 5003, False)])
def test_ce_logits_writes_only_the_gradient_rows(N, V, bf16):
    """Cross-entropy over given logits with a padded gradient buffer: the row
    padding and the guard bytes around the gradient, lse and loss keep their
    pattern (staged and streamed row kernels)."""
    dev = torch.device("cuda:0")
    esz = 2 if bf16 else 4
    ld = (V + 15) // 16 * 16
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([V, N])))
    Z = torch.from_numpy((g.standard_normal((N, V), dtype=np.float32) * 1.3)).to(dev)
    Z = Z.to(torch.bfloat16) if bf16 else Z
    zfull = torch.zeros(N, ld, dtype=Z.dtype, device=dev)
    zfull[:, :V] = Z
    lab = torch.from_numpy(g.integers(0, V, N).astype(np.int32)).to(dev)
    gbuf, graw = _guarded(N * ld * esz, dev)
    gview = graw.view(torch.bfloat16 if bf16 else torch.float32).view(N, ld)[:, :V]
    lbuf, lraw = _guarded(N * 4, dev)
    sbuf, sraw = _guarded(4, dev)
    res = flce.ce_logits(zfull[:, :V], lab, out={"dlogits": gview, "lse": lraw.view(torch.float32),
                                                 "loss": sraw.view(torch.float32)})
    assert flce.check_status(res.status) == flce.FLCE_OK
    for name, b in (("dlogits", gbuf), ("lse", lbuf), ("loss", sbuf)):
        assert _guards_intact(b), name
    pad = graw.view(N, ld * esz)[:, V * esz:].cpu().numpy()
    assert (pad == PATTERN).all()
    assert torch.isfinite(res.dlogits.float()).all()
