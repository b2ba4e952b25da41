"""The library's calls are stream-ordered and allocate nothing, so a whole fused
forward + backward can be captured into a CUDA graph and replayed: replays give
bitwise the results of eager calls, and read the inputs afresh each time."""
import numpy as np
import pytest

import flce_inputs
from flce_testlib import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import linear_cross_entropy_flce_gb300 as flce


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def _alloc(N, D, V, dev):
    return {"loss": torch.empty(1, device=dev), "lse": torch.empty(N, device=dev),
            "dH": torch.empty(N, D, dtype=torch.bfloat16, device=dev),
            "dW": torch.empty(V, D, device=dev)}


@pytest.mark.parametrize("opts", [{}, {"v_chunk": 512, "n_block": 256}])
def test_captured_forward_backward_replays_bitwise(opts):
    wl = flce_inputs.Workload("graph", 700, 256, 3000, 1.0, 0.05, "zipf", 0.1, seed=11)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    N, D, V = wl.N, wl.D, wl.V
    dev = H.device
    ws = torch.empty(flce.workspace_size(N, D, V, flce.make_options(**opts)), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    eager = _alloc(N, D, V, dev)
    flce.forward_backward(H, W, lab, out=eager, workspace=ws, status=st, **opts)
    torch.cuda.synchronize()
    assert flce.check_status(st) == flce.FLCE_OK

    graph_out = _alloc(N, D, V, dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one call on a side stream before capture
        flce.forward_backward(H, W, lab, out=graph_out, workspace=ws, status=st, **opts)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        flce.forward_backward(H, W, lab, out=graph_out, workspace=ws, status=st, **opts)
    for t in graph_out.values():
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert flce.check_status(st) == flce.FLCE_OK
    for k in ("loss", "lse", "dH", "dW"):
        assert torch.equal(_bits(graph_out[k]), _bits(eager[k])), k

    # new inputs written in place: the replay reads them, as an eager call does
    H.copy_(torch.flip(H, dims=[0]))
    lab.copy_(torch.flip(lab, dims=[0]))
    g.replay()
    flce.forward_backward(H, W, lab, out=eager, workspace=torch.empty_like(ws), **opts)
    torch.cuda.synchronize()
    for k in ("loss", "lse", "dH", "dW"):
        assert torch.equal(_bits(graph_out[k]), _bits(eager[k])), k


def test_captured_fp8_step_with_device_quantisation():
    """The FP8 step (quantise H and W on the device, then the FP8 forward + backward
    reading both scales from device memory) holds no host round trip, so it can be
    captured whole; a replay after H changes picks up the new amax and scale."""
    wl = flce_inputs.Workload("graph8", 600, 256, 2500, 1.0, 0.05, "uniform", 0.05, seed=12)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    N, D, V = wl.N, wl.D, wl.V
    dev = H.device
    ws = torch.empty(flce.workspace_size(N, D, V), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    q = {"H8": torch.empty(N, D, dtype=torch.uint8, device=dev),
         "W8": torch.empty(V, D, dtype=torch.uint8, device=dev),
         "sh": torch.empty(2, device=dev), "sw": torch.empty(2, device=dev)}

    def step(out, workspace, status):
        flce.quantize_e4m3(H, q=q["H8"], out=q["sh"])
        flce.quantize_e4m3(W, q=q["W8"], out=q["sw"])
        flce.forward_backward_fp8(q["H8"], q["sh"], q["W8"], q["sw"], lab, H, W, out=out,
                                  workspace=workspace, status=status)

    eager = _alloc(N, D, V, dev)
    step(eager, ws, st)
    torch.cuda.synchronize()
    assert flce.check_status(st) == flce.FLCE_OK
    graph_out = _alloc(N, D, V, dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(graph_out, ws, st)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(graph_out, ws, st)
    for t in graph_out.values():
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert flce.check_status(st) == flce.FLCE_OK
    for k in ("loss", "lse", "dH", "dW"):
        assert torch.equal(_bits(graph_out[k]), _bits(eager[k])), k

    scale_before = q["sh"][0].item()
    H.mul_(2)   # exact in bf16: amax and the scale double
    g.replay()
    torch.cuda.synchronize()
    assert q["sh"][0].item() == 2 * scale_before
    step(eager, torch.empty_like(ws), st)
    torch.cuda.synchronize()
    for k in ("loss", "lse", "dH", "dW"):
        assert torch.equal(_bits(graph_out[k]), _bits(eager[k])), k
