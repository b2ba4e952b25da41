"""flce_forward_noalloc, the forward entry point for callers that cannot
allocate device memory (and so cannot pass a workspace), must give the same
loss and lse as flce_forward, call after call, and after its set-up call it
must take no device memory at all.

Run last on purpose (file name): if it fails, a run stopped at the first
failure has already run every other test. It passes alone in a fresh process
(the first call sets up the library's scratch address) and after the others.
"""
import ctypes

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


def _call(fn, H, W, lab, N, D, V, loss, lse, status, opts=None):
    stream = torch.cuda.current_stream(H.device).cuda_stream
    return fn(H.data_ptr(), W.data_ptr(), lab.data_ptr(), N, D, V,
              ctypes.addressof(opts) if opts is not None else None, loss.data_ptr(),
              lse.data_ptr(), status.data_ptr() if status is not None else None, stream)


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
        rc = _call(fn, H, W, lab, N, D, V, loss, lse, status)
        assert rc == flce.FLCE_OK, flce.status_string(rc)
        assert flce.check_status(status) == flce.FLCE_OK
        assert flce.check_status(ref.status) == flce.FLCE_OK
        a, b = float(loss.item()), float(ref.loss.item())
        assert abs(a - b) <= TOL_LOSS_REL * abs(b)
        assert float((lse - ref.lse).abs().max()) <= TOL_LSE_ABS


def test_forward_noalloc_takes_no_device_memory_after_set_up():
    """After the set-up call and one warm-up call, a further call leaves the
    device's free memory (cudaMemGetInfo) exactly where it was."""
    flce, fn = _noalloc()
    assert fn(None, None, None, 0, 0, 0, None, None, None, None, None) == flce.FLCE_OK
    N, D, V = 900, 256, 4000
    wl = flce_inputs.Workload("noalloc_mem", N, D, V, 1.0, 0.05, "uniform", 0.1, seed=23)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    loss = torch.empty(1, dtype=torch.float32, device=H.device)
    lse = torch.empty(N, dtype=torch.float32, device=H.device)
    status = torch.zeros(1, dtype=torch.int32, device=H.device)
    assert _call(fn, H, W, lab, N, D, V, loss, lse, status) == flce.FLCE_OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(H.device)[0]
    for _ in range(3):
        assert _call(fn, H, W, lab, N, D, V, loss, lse, status) == flce.FLCE_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(H.device)[0] == free0
    assert flce.check_status(status) == flce.FLCE_OK


def test_forward_noalloc_large_token_count_and_explicit_split_kept():
    """A million tokens fit in the static scratch with the planned vocabulary
    ranges (the result matches flce_forward); the same problem with an explicit
    v_splits whose partials do not fit is rejected instead of being changed."""
    flce, fn = _noalloc()
    N, D, V = 1_000_000, 8, 1024
    wl = flce_inputs.Workload("noalloc_big", N, D, V, 1.0, 0.5, "uniform", 0.1, seed=24)
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H, W, lab = to_device(Hb, Wb, y)
    loss = torch.empty(1, dtype=torch.float32, device=H.device)
    lse = torch.empty(N, dtype=torch.float32, device=H.device)
    status = torch.zeros(1, dtype=torch.int32, device=H.device)
    assert _call(fn, H, W, lab, N, D, V, loss, lse, status) == flce.FLCE_OK
    ref = flce.forward(H, W, lab)
    assert flce.check_status(status) == flce.FLCE_OK and flce.check_status(ref.status) == flce.FLCE_OK
    assert abs(float(loss.item()) - float(ref.loss.item())) <= TOL_LOSS_REL * abs(float(ref.loss.item()))
    assert float((lse - ref.lse).abs().max()) <= TOL_LSE_ABS
    one = flce.make_options(v_splits=1)     # 8 B of partials per token: fits
    assert _call(fn, H, W, lab, N, D, V, loss, lse, status, one) == flce.FLCE_OK
    assert flce.check_status(status) == flce.FLCE_OK
    four = flce.make_options(v_splits=4)    # 32 B of partials per token: does not fit
    assert flce.forward_workspace_size(N, D, V, four) > 32 << 20
    assert _call(fn, H, W, lab, N, D, V, loss, lse, status, four) == flce.FLCE_ERR_WORKSPACE


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
    rc = _call(fn, H, W, lab, N, D, V, loss, lse, None)
    assert rc == flce.FLCE_ERR_WORKSPACE
