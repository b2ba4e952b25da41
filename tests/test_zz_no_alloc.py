"""flce_forward_noalloc, the forward entry point for callers that cannot
allocate device memory (and so cannot pass a workspace), must give the same
loss and lse as flce_forward, call after call.

Run last on purpose (file name): if it fails, a run stopped at the first
failure has already run every other test. It passes alone in a fresh process
(the first call sets up the library's scratch address) and after the others.
"""
import ctypes

import numpy as np
import pytest

import flce_inputs
from flce_testlib import TOL_LOSS_REL, TOL_LSE_ABS, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _noalloc():
    import linear_cross_entropy_flce_gb300 as flce
    fn = flce.lib.flce_forward_noalloc
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    fn.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, vp, vp]
    fn.restype = ctypes.c_int
    return flce, fn


def test_forward_noalloc_matches_forward_on_two_calls_in_a_row():
    flce, fn = _noalloc()
    # Two different problems back to back: the second call must not see the
    # first call's leftovers in the shared scratch array.
    for seed, (N, D, V) in [(21, (1000, 512, 5000)), (22, (777, 256, 3000))]:
        wl = flce_inputs.Workload("noalloc", N, D, V, 1.0, 0.05, "uniform", 0.1, seed=seed)
        Hb, Wb, y = flce_inputs.make_inputs(wl)
        H, W, lab = to_device(Hb, Wb, y)
        ref = flce.forward(H, W, lab)
        loss = torch.empty(1, dtype=torch.float32, device=H.device)
        lse = torch.empty(N, dtype=torch.float32, device=H.device)
        status = torch.full((1,), -1, dtype=torch.int32, device=H.device)
        stream = torch.cuda.current_stream(H.device).cuda_stream
        rc = fn(H.data_ptr(), W.data_ptr(), lab.data_ptr(), N, D, V, None, loss.data_ptr(),
                lse.data_ptr(), status.data_ptr(), stream)
        assert rc == flce.FLCE_OK, flce.status_string(rc)
        assert flce.check_status(status) == flce.FLCE_OK
        assert flce.check_status(ref.status) == flce.FLCE_OK
        a, b = float(loss.item()), float(ref.loss.item())
        assert abs(a - b) <= TOL_LOSS_REL * abs(b)
        assert float((lse - ref.lse).abs().max()) <= TOL_LSE_ABS


def test_forward_noalloc_rejects_problems_beyond_its_scratch():
    flce, fn = _noalloc()
    # about 20 bytes of scratch per token: 2M tokens need ~40 MB > 32 MiB.
    # The buffers are real (and small, D = 8) so that nothing could go astray.
    N, D, V = 2_000_000, 8, 256
    dev = torch.device("cuda:0")
    H = torch.zeros(N, D, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(V, D, dtype=torch.bfloat16, device=dev)
    lab = torch.zeros(N, dtype=torch.int32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    rc = fn(H.data_ptr(), W.data_ptr(), lab.data_ptr(), N, D, V, None, loss.data_ptr(),
            lse.data_ptr(), None, torch.cuda.current_stream(dev).cuda_stream)
    assert rc == flce.FLCE_ERR_WORKSPACE
