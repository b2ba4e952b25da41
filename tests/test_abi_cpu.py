"""The C-ABI library loads without a GPU, exports every function that
include/flce.h declares, and rejects bad arguments on the host before any
device work (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import linear_cross_entropy_flce_gb300 as flce
from linear_cross_entropy_flce_gb300 import _binding

HEADER = _binding.HEADER_PATH


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert names == sorted(["flce_default_options", "flce_workspace_size",
                            "flce_forward_workspace_size", "flce_get_plan",
                            "flce_forward_backward", "flce_forward", "flce_forward_noalloc",
                            "flce_ce_workspace_size", "flce_ce_logits", "flce_forward_fp8",
                            "flce_forward_backward_fp8", "flce_quantize_e4m3",
                            "flce_forward_shard", "flce_backward_shard",
                            "flce_scale_grads",
                            "flce_check_status", "flce_status_string"])


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(flce.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_default_options():
    o = flce.make_options()
    assert (o.ignore_index, o.reduction, o.grad_scale, o.normalizer, o.dw_dtype) == (-100, 0, 1.0, 0.0, 0)
    assert (o.v_splits, o.n_block, o.v_chunk, o.timeout_ns) == (0, 0, 0, 0)
    assert ctypes.sizeof(flce.Options) == 64
    assert o.trace_events is None and o.trace_capacity == 0 and o.reserved == 0


def test_workspace_is_far_below_logits():
    # The bound is one G chunk (at most 16384 vocabulary ids x at most 256 MiB)
    # plus small per-token arrays and one fp32 dH block; at tile-sized problems
    # the 256 x 256 tile rounding dominates instead.
    assert flce.workspace_size(64, 128, 1000) < 1 << 20
    for N, D, V, frac in [(4096, 2048, 32000, 0.35), (8192, 4096, 128256, 0.11),
                          (16384, 3584, 152064, 0.05), (32768, 4096, 128256, 0.03)]:
        ws = flce.workspace_size(N, D, V)
        assert 0 < ws < N * V * 4 * frac, (N, D, V, ws)
        assert ws < 600 << 20


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("N,D,V,S", [(1_000_000, 4096, 128256, 1), (8192, 4096, 128256, 2),
                                     (300, 200, 1500, 3)])
def test_forward_workspace_matches_the_header_formula(N, D, V, S):
    """flce_forward_workspace_size against the formula include/flce.h states:
    align256(8 S 256 ceil(N/256)) + 3 align256(4 N) + 256, independent of D."""
    want = _align256(8 * S * 256 * (-(-N // 256))) + 3 * _align256(4 * N) + 256
    opts = flce.make_options(v_splits=S)
    assert flce.forward_workspace_size(N, D, V, opts) == want
    assert flce.forward_workspace_size(N, 8 * D, V, opts) == want
    assert flce.forward_workspace_size(N, D, V, opts) < flce.workspace_size(N, D, V, opts)


def test_noalloc_limit_stated_in_the_header():
    """The no-workspace entry point's scratch is 32 MiB: with S = 1, about 20 bytes
    per token fit about 1.6 million tokens, whatever D and V."""
    one = flce.make_options(v_splits=1)
    assert flce.forward_workspace_size(1_600_000, 4096, 128256, one) <= 32 << 20
    assert flce.forward_workspace_size(1_700_000, 4096, 128256, one) > 32 << 20
    assert flce.forward_workspace_size(2_000_000, 8, 256, one) > 32 << 20


def test_workspace_grows_with_requested_chunk():
    a = flce.workspace_size(8192, 4096, 128256, flce.make_options(v_chunk=4096, n_block=8192))
    b = flce.workspace_size(8192, 4096, 128256, flce.make_options(v_chunk=16384, n_block=8192))
    assert b - a == pytest.approx(8192 * (16384 - 4096) * 2, rel=0.01)


@pytest.mark.parametrize("kw,code", [
    (dict(N=0, D=128, V=10), flce.FLCE_ERR_SHAPE),
    (dict(N=8, D=0, V=10), flce.FLCE_ERR_SHAPE),
    (dict(N=8, D=128, V=0), flce.FLCE_ERR_SHAPE),
    (dict(N=8, D=100, V=10), flce.FLCE_ERR_ALIGN),
])
def test_workspace_size_rejects_bad_shapes(kw, code):
    out = ctypes.c_size_t()
    assert flce.lib.flce_workspace_size(kw["N"], kw["D"], kw["V"], None, ctypes.byref(out)) == code


@pytest.mark.parametrize("opt,code", [
    (dict(reduction=7), flce.FLCE_ERR_OPTION),
    (dict(dw_dtype=3), flce.FLCE_ERR_OPTION),
    (dict(v_chunk=300), flce.FLCE_ERR_OPTION),
    (dict(n_block=100), flce.FLCE_ERR_OPTION),
    (dict(timeout_ns=-1), flce.FLCE_ERR_OPTION),
    (dict(trace_capacity=3), flce.FLCE_ERR_OPTION),
    (dict(reserved=1), flce.FLCE_ERR_OPTION),
])
def test_workspace_size_rejects_bad_options(opt, code):
    o = flce.make_options()
    for k, v in opt.items():
        setattr(o, k, v)
    out = ctypes.c_size_t()
    assert flce.lib.flce_workspace_size(64, 128, 1000, ctypes.byref(o), ctypes.byref(out)) == code


def _call(H=0x1000, W=0x2000, y=0x3000, N=64, D=128, V=1000, loss=0x4000, ws=0x5000,
          ws_bytes=1 << 30, status=None, opts=None):
    return flce.lib.flce_forward_backward(H, W, y, N, D, V, ctypes.byref(opts) if opts else None,
                                          loss, None, None, None, ws, ws_bytes, status, None)


def test_host_rejections_happen_before_device_work():
    assert _call(H=None) == flce.FLCE_ERR_NULL
    assert _call(W=None) == flce.FLCE_ERR_NULL
    assert _call(y=None) == flce.FLCE_ERR_NULL
    assert _call(loss=None) == flce.FLCE_ERR_NULL
    assert _call(ws=None) == flce.FLCE_ERR_NULL
    assert _call(N=-1) == flce.FLCE_ERR_SHAPE
    assert _call(D=12) == flce.FLCE_ERR_ALIGN
    assert _call(H=0x1008) == flce.FLCE_ERR_ALIGN
    assert _call(ws=0x5004) == flce.FLCE_ERR_ALIGN
    o = flce.make_options()
    o.reduction = 5
    assert _call(opts=o) == flce.FLCE_ERR_OPTION


def test_plan_rejections_before_device_query():
    from linear_cross_entropy_flce_gb300._binding import PlanInfo
    info = PlanInfo()
    assert flce.lib.flce_get_plan(64, 128, 1000, None, 1, 1, None) == flce.FLCE_ERR_NULL
    assert flce.lib.flce_get_plan(0, 128, 1000, None, 1, 1, ctypes.byref(info)) == flce.FLCE_ERR_SHAPE
    assert flce.lib.flce_get_plan(64, 12, 1000, None, 1, 1, ctypes.byref(info)) == flce.FLCE_ERR_ALIGN


def test_ce_logits_host_rejections():
    f = flce.lib.flce_ce_logits
    ws = ctypes.c_size_t()
    assert flce.lib.flce_ce_workspace_size(8, 100, None, ctypes.byref(ws)) == flce.FLCE_OK
    assert ws.value >= 2 * 8 * 4

    def call(logits=0x1000, dtype=0, ld=128, y=0x2000, N=8, V=100, loss=0x3000, dl=None,
             dld=0, w=0x4000, opts=None):
        return f(logits, dtype, ld, y, N, V, ctypes.byref(opts) if opts else None, loss, None,
                 dl, dld, w, 1 << 20, None, None)

    assert call(logits=None) == flce.FLCE_ERR_NULL
    assert call(N=0) == flce.FLCE_ERR_SHAPE
    assert call(ld=99) == flce.FLCE_ERR_SHAPE
    assert call(ld=102) == flce.FLCE_ERR_ALIGN          # 408-byte rows
    assert call(dtype=1, ld=100) == flce.FLCE_ERR_ALIGN  # 200-byte rows
    assert call(dtype=7) == flce.FLCE_ERR_OPTION
    assert call(dl=0x1000, dld=256) == flce.FLCE_ERR_OPTION  # in place with another stride
    o = flce.make_options(reduction="none")
    assert call(dl=0x8000, dld=128, opts=o) == flce.FLCE_ERR_OPTION


def test_fp8_host_rejections():
    f = flce.lib.flce_forward_fp8
    ok = dict(H8=0x1000, sh=0x8000, W8=0x2000, sw=0x8004, y=0x3000, N=64, D=128, V=1000,
              loss=0x4000, ws=0x5000)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["H8"], a["sh"], a["W8"], a["sw"], a["y"], a["N"], a["D"], a["V"], None,
                 a["loss"], None, a["ws"], 1 << 30, None, None)

    assert call(H8=None) == flce.FLCE_ERR_NULL
    assert call(W8=None) == flce.FLCE_ERR_NULL
    assert call(D=136) == flce.FLCE_ERR_ALIGN      # D % 16 != 0 for E4M3 rows
    assert call(H8=0x1004) == flce.FLCE_ERR_ALIGN
    assert call(sh=None) == flce.FLCE_ERR_NULL     # scales are device fp32 scalars
    assert call(sw=None) == flce.FLCE_ERR_NULL
    assert call(sh=0x8002) == flce.FLCE_ERR_ALIGN
    g = flce.lib.flce_forward_backward_fp8
    # the gradient products need the bf16 operands
    assert g(0x1000, 0x8000, 0x2000, 0x8004, None, None, 0x3000, 64, 128, 1000, None, 0x4000,
             None, 0x6000, 0x7000, 0x5000, 1 << 30, None, None) == flce.FLCE_ERR_NULL


def test_shard_host_rejections():
    f = flce.lib.flce_forward_shard
    ok = dict(H=0x1000, W=0x2000, y=0x3000, N=64, D=128, V=500, off=500, Vt=1000, m=0x4000,
              s=0x5000, zt=0x6000, ws=0x7000)

    def fwd(**kw):
        a = dict(ok, **kw)
        return f(a["H"], a["W"], a["y"], a["N"], a["D"], a["V"], a["off"], a["Vt"], None, a["m"],
                 a["s"], a["zt"], a["ws"], 1 << 30, None, None)

    assert fwd(m=None) == flce.FLCE_ERR_NULL
    assert fwd(zt=None) == flce.FLCE_ERR_NULL
    assert fwd(off=-1) == flce.FLCE_ERR_SHAPE
    assert fwd(off=501) == flce.FLCE_ERR_SHAPE     # past the whole vocabulary
    assert fwd(Vt=0) == flce.FLCE_ERR_SHAPE
    assert fwd(s=0x5002) == flce.FLCE_ERR_ALIGN
    g = flce.lib.flce_backward_shard

    def bwd(lse=0x8000, dh=0x9000, dw=0xA000, off=500):
        return g(0x1000, 0x2000, 0x3000, 64, 128, 500, off, 1000, None, lse, dh, dw, 0x7000,
                 1 << 30, None, None)

    assert bwd(lse=None) == flce.FLCE_ERR_NULL
    assert bwd(dh=None, dw=None) == flce.FLCE_ERR_NULL
    assert bwd(dh=0x9008) == flce.FLCE_ERR_ALIGN   # TMA base of the fp32 dH part
    assert bwd(off=600) == flce.FLCE_ERR_SHAPE


def test_quantize_e4m3_host_rejections():
    f = flce.lib.flce_quantize_e4m3
    assert f(None, 64, 0x2000, 0x3000, None) == flce.FLCE_ERR_NULL
    assert f(0x1000, 64, None, 0x3000, None) == flce.FLCE_ERR_NULL
    assert f(0x1000, 64, 0x2000, None, None) == flce.FLCE_ERR_NULL
    assert f(0x1000, 0, 0x2000, 0x3000, None) == flce.FLCE_ERR_SHAPE
    assert f(0x1000, 12, 0x2000, 0x3000, None) == flce.FLCE_ERR_ALIGN   # n % 8 != 0
    assert f(0x1008, 64, 0x2000, 0x3000, None) == flce.FLCE_ERR_ALIGN
    assert f(0x1000, 64, 0x2008, 0x3000, None) == flce.FLCE_ERR_ALIGN
    assert f(0x1000, 64, 0x2000, 0x3004, None) == flce.FLCE_ERR_ALIGN


def test_scale_grads_host_rejections():
    f = flce.lib.flce_scale_grads
    assert f(0x1000, 8, None, 0, 0, None, None) == flce.FLCE_ERR_NULL
    assert f(None, 8, None, 0, 0, 0x2000, None) == flce.FLCE_ERR_NULL
    assert f(0x1000, 4, None, 0, 0, 0x2000, None) == flce.FLCE_ERR_ALIGN   # 8 bytes of bf16
    assert f(0x1000, 8, 0x3000, 8, 5, 0x2000, None) == flce.FLCE_ERR_OPTION
    assert f(0x1000, -8, None, 0, 0, 0x2000, None) == flce.FLCE_ERR_SHAPE


def test_status_strings():
    for code in range(0, 10):
        assert flce.status_string(code) and flce.status_string(code) != "unknown status"
    assert flce.status_string(1234) == "unknown status"


def test_header_compiles_as_c_and_links(tmp_path):
    """A plain C99 program includes include/flce.h, links libflce.so and calls the
    entry points that need no GPU (tests/abi_c_check.c)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    libdir = os.path.dirname(_binding.LIB_PATH)
    exe = str(tmp_path / "abi_c_check")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER),
           os.path.join(here, "abi_c_check.c"), "-L", libdir, "-lflce",
           "-Wl,-rpath," + libdir, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
