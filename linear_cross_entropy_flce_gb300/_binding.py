"""ctypes binding of libflce.so (include/flce.h): argument marshalling only.

Every computation happens in the library's CUDA kernels. PyTorch is used here
only for device memory, streams and tensor metadata. If the library has not
been built, importing this module raises ImportError: there is no fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libflce.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "flce.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
        "(fused linear cross-entropy has no CPU or PyTorch fallback)")

lib = ctypes.CDLL(LIB_PATH)

FLCE_OK = 0
FLCE_ERR_NULL = 1
FLCE_ERR_SHAPE = 2
FLCE_ERR_ALIGN = 3
FLCE_ERR_WORKSPACE = 4
FLCE_ERR_OPTION = 5
FLCE_ERR_CUDA = 6
FLCE_ERR_DEVICE = 7
FLCE_ERR_LABEL_RANGE = 8
FLCE_ERR_TIMEOUT = 9

REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}
DW_DTYPES = {"float32": 0, "bfloat16": 1}


class Options(ctypes.Structure):
    _fields_ = [
        ("ignore_index", ctypes.c_int32),
        ("reduction", ctypes.c_int32),
        ("grad_scale", ctypes.c_float),
        ("normalizer", ctypes.c_float),
        ("dw_dtype", ctypes.c_int32),
        ("v_splits", ctypes.c_int32),
        ("n_block", ctypes.c_int64),
        ("v_chunk", ctypes.c_int64),
        ("timeout_ns", ctypes.c_int64),
        ("trace_events", ctypes.c_void_p),
        ("trace_capacity", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("n_block", ctypes.c_int64),
        ("v_chunk", ctypes.c_int64),
        ("n_blocks", ctypes.c_int32),
        ("n_chunks", ctypes.c_int32),
        ("v_splits", ctypes.c_int32),
        ("kernel_launches", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_size_t),
        ("plan_bytes", ctypes.c_size_t),
    ]


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
lib.flce_default_options.argtypes = [ctypes.POINTER(Options)]
lib.flce_default_options.restype = None
lib.flce_workspace_size.argtypes = [_i64, _i64, _i64, ctypes.POINTER(Options),
                                    ctypes.POINTER(ctypes.c_size_t)]
lib.flce_workspace_size.restype = ctypes.c_int
lib.flce_forward_workspace_size.argtypes = [_i64, _i64, _i64, ctypes.POINTER(Options),
                                            ctypes.POINTER(ctypes.c_size_t)]
lib.flce_forward_workspace_size.restype = ctypes.c_int
lib.flce_forward_noalloc.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.POINTER(Options),
                                     _vp, _vp, _vp, _vp]
lib.flce_forward_noalloc.restype = ctypes.c_int
lib.flce_get_plan.argtypes = [_i64, _i64, _i64, ctypes.POINTER(Options), ctypes.c_int32,
                              ctypes.c_int32, ctypes.POINTER(PlanInfo)]
lib.flce_get_plan.restype = ctypes.c_int
lib.flce_forward_backward.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.POINTER(Options),
                                      _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]
lib.flce_forward_backward.restype = ctypes.c_int
lib.flce_forward.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.POINTER(Options),
                             _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]
lib.flce_forward.restype = ctypes.c_int
lib.flce_ce_workspace_size.argtypes = [_i64, _i64, ctypes.POINTER(Options),
                                       ctypes.POINTER(ctypes.c_size_t)]
lib.flce_ce_workspace_size.restype = ctypes.c_int
lib.flce_ce_logits.argtypes = [_vp, ctypes.c_int32, _i64, _vp, _i64, _i64, ctypes.POINTER(Options),
                               _vp, _vp, _vp, _i64, _vp, ctypes.c_size_t, _vp, _vp]
lib.flce_ce_logits.restype = ctypes.c_int
lib.flce_forward_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                 ctypes.POINTER(Options), _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]
lib.flce_forward_fp8.restype = ctypes.c_int
lib.flce_forward_backward_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                          ctypes.POINTER(Options), _vp, _vp, _vp, _vp, _vp,
                                          ctypes.c_size_t, _vp, _vp]
lib.flce_forward_backward_fp8.restype = ctypes.c_int
lib.flce_scale_grads.argtypes = [_vp, _i64, _vp, _i64, ctypes.c_int32, _vp, _vp]
lib.flce_scale_grads.restype = ctypes.c_int
lib.flce_forward_shard.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                   ctypes.POINTER(Options), _vp, _vp, _vp, _vp, ctypes.c_size_t,
                                   _vp, _vp]
lib.flce_forward_shard.restype = ctypes.c_int
lib.flce_backward_shard.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                    ctypes.POINTER(Options), _vp, _vp, _vp, _vp, ctypes.c_size_t,
                                    _vp, _vp]
lib.flce_backward_shard.restype = ctypes.c_int
lib.flce_quantize_e4m3.argtypes = [_vp, _i64, _vp, _vp, _vp]
lib.flce_quantize_e4m3.restype = ctypes.c_int
lib.flce_check_status.argtypes = [_vp, _vp]
lib.flce_check_status.restype = ctypes.c_int
lib.flce_status_string.argtypes = [ctypes.c_int]
lib.flce_status_string.restype = ctypes.c_char_p


class FLCEError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        super().__init__(f"{where}: flce error {code}: {status_string(code)}")


def status_string(code: int) -> str:
    return lib.flce_status_string(int(code)).decode()


def make_options(*, ignore_index: int = -100, reduction: str = "mean", grad_scale: float = 1.0,
                 normalizer: float = 0.0, dw_dtype: str = "float32", v_splits: int = 0,
                 n_block: int = 0, v_chunk: int = 0, timeout_ns: int = 0,
                 trace_events=None) -> Options:
    """trace_events: optional sequence of torch.cuda.Event (or raw cudaEvent_t
    integers); the library records event 0 before its first kernel and event k
    after its k-th kernel."""
    o = Options()
    lib.flce_default_options(ctypes.byref(o))
    o.ignore_index = int(ignore_index)
    o.reduction = REDUCTIONS[reduction]
    o.grad_scale = float(grad_scale)
    o.normalizer = float(normalizer)
    o.dw_dtype = DW_DTYPES[dw_dtype]
    o.v_splits = int(v_splits)
    o.n_block = int(n_block)
    o.v_chunk = int(v_chunk)
    o.timeout_ns = int(timeout_ns)
    if trace_events is not None:
        handles = [int(getattr(e, "cuda_event", e)) for e in trace_events]
        arr = (ctypes.c_void_p * len(handles))(*handles)
        o._trace_keepalive = arr
        o.trace_events = ctypes.cast(arr, ctypes.c_void_p)
        o.trace_capacity = len(handles)
    return o


def workspace_size(N: int, D: int, V: int, opts: Optional[Options] = None) -> int:
    out = ctypes.c_size_t(0)
    rc = lib.flce_workspace_size(N, D, V, ctypes.byref(opts) if opts is not None else None,
                                 ctypes.byref(out))
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_workspace_size")
    return int(out.value)


def forward_workspace_size(N: int, D: int, V: int, opts: Optional[Options] = None) -> int:
    """Workspace bytes of the forward-only calls (flce_forward_workspace_size)."""
    out = ctypes.c_size_t(0)
    rc = lib.flce_forward_workspace_size(N, D, V, ctypes.byref(opts) if opts is not None else None,
                                         ctypes.byref(out))
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_forward_workspace_size")
    return int(out.value)


def get_plan(N: int, D: int, V: int, opts: Optional[Options] = None, want_dh: bool = True,
             want_dw: bool = True) -> dict:
    """The plan flce_forward_backward uses on the current device (needs a GPU)."""
    info = PlanInfo()
    rc = lib.flce_get_plan(N, D, V, ctypes.byref(opts) if opts is not None else None,
                           int(want_dh), int(want_dw), ctypes.byref(info))
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_get_plan")
    return {k: getattr(info, k) for k, _ in PlanInfo._fields_}


@dataclasses.dataclass
class Result:
    loss: "object"           # torch float32 [1]
    lse: "object"            # torch float32 [N]
    dH: "object" = None      # torch bfloat16 [N, D] or None
    dW: "object" = None      # torch float32/bfloat16 [V, D] or None
    status: "object" = None  # torch int32 [1] (device status word)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _check_inputs(H, W, labels):
    import torch
    if not (H.is_cuda and W.is_cuda and labels.is_cuda):
        raise ValueError("H, W and labels must be CUDA tensors")
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("H and W must be bfloat16")
    if labels.dtype != torch.int32:
        raise TypeError("labels must be int32")
    if H.dim() != 2 or W.dim() != 2 or labels.dim() != 1:
        raise ValueError("H must be [N, D], W [V, D], labels [N]")
    if not (H.is_contiguous() and W.is_contiguous() and labels.is_contiguous()):
        raise ValueError("H, W and labels must be contiguous")
    N, D = H.shape
    V, D2 = W.shape
    if D2 != D or labels.shape[0] != N:
        raise ValueError("shape mismatch between H, W and labels")
    return N, D, V


def forward_backward(H, W, labels, *, need_dh: bool = True, need_dw: bool = True,
                     out: Optional[dict] = None, workspace=None, status=None, stream=None,
                     **options) -> Result:
    """Loss, lse, dH and dW of fused linear cross-entropy via flce_forward_backward.

    options: ignore_index, reduction ("mean"/"sum"), grad_scale, normalizer,
    dw_dtype ("float32"/"bfloat16"), v_splits, n_block, v_chunk, timeout_ns.
    `out` may hold preallocated "loss", "lse", "dH", "dW" tensors.
    """
    import torch
    N, D, V = _check_inputs(H, W, labels)
    opts = make_options(**options)
    dev = H.device
    out = dict(out or {})
    loss = out.get("loss")
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = out.get("lse")
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    dH = out.get("dH")
    if dH is None and need_dh:
        dH = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
    dW = out.get("dW")
    if dW is None and need_dw:
        dt = torch.float32 if options.get("dw_dtype", "float32") == "float32" else torch.bfloat16
        dW = torch.empty(V, D, dtype=dt, device=dev)
    ws_bytes = workspace_size(N, D, V, opts)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.flce_forward_backward(_ptr(H), _ptr(W), _ptr(labels), N, D, V, ctypes.byref(opts),
                                   _ptr(loss), _ptr(lse), _ptr(dH) if need_dh else None,
                                   _ptr(dW) if need_dw else None, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(status),
                                   stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_forward_backward")
    return Result(loss, lse, dH if need_dh else None, dW if need_dw else None, status)


def forward(H, W, labels, *, out: Optional[dict] = None, workspace=None, status=None,
            stream=None, **options) -> Result:
    """Loss and lse only, via flce_forward. With reduction="none" the loss is
    the per-token loss [N] (0 for ignored tokens)."""
    import torch
    N, D, V = _check_inputs(H, W, labels)
    opts = make_options(**options)
    dev = H.device
    out = dict(out or {})
    loss = out.get("loss")
    if loss is None:
        n_loss = N if options.get("reduction") == "none" else 1
        loss = torch.empty(n_loss, dtype=torch.float32, device=dev)
    lse = out.get("lse")
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(forward_workspace_size(N, D, V, opts), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.flce_forward(_ptr(H), _ptr(W), _ptr(labels), N, D, V, ctypes.byref(opts),
                          _ptr(loss), _ptr(lse), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _ptr(status), stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_forward")
    return Result(loss, lse, None, None, status)


def forward_noalloc(H, W, labels, *, out: Optional[dict] = None, status=None, stream=None,
                    **options) -> Result:
    """Loss and lse via flce_forward_noalloc: the library's own static scratch
    instead of a workspace (for callers that cannot allocate at call time)."""
    import torch
    N, D, V = _check_inputs(H, W, labels)
    opts = make_options(**options)
    dev = H.device
    out = dict(out or {})
    loss = out.get("loss")
    if loss is None:
        loss = torch.empty(N if options.get("reduction") == "none" else 1, dtype=torch.float32,
                           device=dev)
    lse = out.get("lse")
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.flce_forward_noalloc(_ptr(H), _ptr(W), _ptr(labels), N, D, V, ctypes.byref(opts),
                                  _ptr(loss), _ptr(lse), _ptr(status), stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_forward_noalloc")
    return Result(loss, lse, None, None, status)


def noalloc_setup() -> None:
    """The set-up call of flce_forward_noalloc on the current device (creates the
    library's static scratch there and looks up its address)."""
    rc = lib.flce_forward_noalloc(None, None, None, 0, 0, 0, None, None, None, None, None)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_forward_noalloc set-up")


@dataclasses.dataclass
class ShardForward:
    m: object        # fp32 [N]: max over the shard's ids of z_iv
    s: object        # fp32 [N]: sum over the shard's ids of exp(z_iv - m_i)
    zt: object       # fp32 [N]: target logit if the label lies in the shard, else 0
    status: object


def forward_shard(H, W_shard, labels, v_offset: int, V_total: int, *, out: Optional[dict] = None,
                  workspace=None, status=None, stream=None, **options) -> ShardForward:
    """flce_forward_shard: the per-token (m, s, zt) of vocabulary rows
    [v_offset, v_offset + len(W_shard)) of a V_total-id vocabulary (labels are
    ids of the whole vocabulary)."""
    import torch
    N, D, V = _check_inputs(H, W_shard, labels)
    opts = make_options(**options)
    dev = H.device
    out = dict(out or {})
    m, s_, zt = (out.get(k) if out.get(k) is not None else
                 torch.empty(N, dtype=torch.float32, device=dev) for k in ("m", "s", "zt"))
    if workspace is None:
        workspace = torch.empty(forward_workspace_size(N, D, V, opts), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.flce_forward_shard(_ptr(H), _ptr(W_shard), _ptr(labels), N, D, V, int(v_offset),
                                int(V_total), ctypes.byref(opts), _ptr(m), _ptr(s_), _ptr(zt),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _ptr(status), stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_forward_shard")
    return ShardForward(m, s_, zt, status)


def backward_shard(H, W_shard, labels, lse, v_offset: int, V_total: int, *, need_dh: bool = True,
                   need_dw: bool = True, out: Optional[dict] = None, workspace=None, status=None,
                   stream=None, **options) -> Result:
    """flce_backward_shard: from the combined lse, the shard's fp32 part of dH
    (summed over the shards by the caller) and its rows of dW. Returns a Result
    whose loss is None and whose dH is the fp32 part."""
    import torch
    N, D, V = _check_inputs(H, W_shard, labels)
    if not (lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous() and lse.numel() == N):
        raise ValueError("lse must be a contiguous CUDA float32 tensor of N values")
    opts = make_options(**options)
    dev = H.device
    out = dict(out or {})
    dH = out.get("dH")
    if dH is None and need_dh:
        dH = torch.empty(N, D, dtype=torch.float32, device=dev)
    dW = out.get("dW")
    if dW is None and need_dw:
        dt = torch.float32 if options.get("dw_dtype", "float32") == "float32" else torch.bfloat16
        dW = torch.empty(V, D, dtype=dt, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_size(N, D, V, opts), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.flce_backward_shard(_ptr(H), _ptr(W_shard), _ptr(labels), N, D, V, int(v_offset),
                                 int(V_total), ctypes.byref(opts), _ptr(lse),
                                 _ptr(dH) if need_dh else None, _ptr(dW) if need_dw else None,
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _ptr(status), stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_backward_shard")
    return Result(None, lse, dH if need_dh else None, dW if need_dw else None, status)


def ce_logits(logits, labels, *, need_grad: bool = True, in_place: bool = False,
              out: Optional[dict] = None, workspace=None, status=None, stream=None,
              **options) -> Result:
    """Cross-entropy over given logits [N, V] (fp32 or bf16) via flce_ce_logits.
    Returns Result(loss, lse, dH=None, dW=None) with the gradient in
    result.dlogits (the logits tensor itself when in_place)."""
    import torch
    if not (logits.is_cuda and labels.is_cuda):
        raise ValueError("logits and labels must be CUDA tensors")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [N, V] with unit column stride")
    if logits.dtype not in (torch.float32, torch.bfloat16) or labels.dtype != torch.int32:
        raise TypeError("logits float32/bfloat16, labels int32")
    N, V = logits.shape
    ld = logits.stride(0)
    dtype = 1 if logits.dtype == torch.bfloat16 else 0
    opts = make_options(**options)
    dev = logits.device
    out = dict(out or {})
    loss = out.get("loss")
    if loss is None:
        loss = torch.empty(N if options.get("reduction") == "none" else 1, dtype=torch.float32,
                           device=dev)
    lse = out.get("lse")
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    grad = None
    if need_grad:
        grad = logits if in_place else out.get("dlogits")
        if grad is None:   # same (padded) row stride as the logits
            grad = torch.empty_strided((N, V), (ld, 1), dtype=logits.dtype, device=dev)
    size = ctypes.c_size_t(0)
    rc = lib.flce_ce_workspace_size(N, V, ctypes.byref(opts), ctypes.byref(size))
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_ce_workspace_size")
    if workspace is None:
        workspace = torch.empty(int(size.value), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.flce_ce_logits(_ptr(logits), dtype, ld, _ptr(labels), N, V, ctypes.byref(opts),
                            _ptr(loss), _ptr(lse), _ptr(grad), grad.stride(0) if grad is not None else 0,
                            _ptr(workspace), workspace.numel(), _ptr(status), stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_ce_logits")
    r = Result(loss, lse, None, None, status)
    r.dlogits = grad
    return r


def _device_scale(scale, dev):
    """A per-tensor scale as a device fp32 scalar: a CUDA float32 tensor whose first
    element is the scale (e.g. out[0] of quantize_e4m3), or a Python number."""
    import torch
    if isinstance(scale, torch.Tensor):
        if not (scale.is_cuda and scale.dtype == torch.float32 and scale.numel() >= 1
                and scale.is_contiguous()):
            raise TypeError("a scale tensor must be a contiguous CUDA float32 tensor")
        return scale
    return torch.tensor([float(scale)], dtype=torch.float32, device=dev)


def quantize_e4m3(x, *, out=None, q=None, stream=None):
    """Per-tensor E4M3 quantisation of a bf16 CUDA tensor on the device via
    flce_quantize_e4m3: returns (q uint8 with x's shape, out float32[2] holding
    [scale, amax]); out[0:1] serves directly as a scale of the FP8 entry points."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise TypeError("x must be a contiguous bf16 CUDA tensor")
    dev = x.device
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(2, dtype=torch.float32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.flce_quantize_e4m3(_ptr(x), x.numel(), _ptr(q), _ptr(out), stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_quantize_e4m3")
    return q, out


def forward_backward_fp8(H8, scale_h, W8, scale_w, labels, H=None, W=None, *,
                         need_dh: bool = True, need_dw: bool = True, out: Optional[dict] = None,
                         workspace=None, status=None, stream=None, **options) -> Result:
    """FP8 operand variant (flce_forward_backward_fp8, or flce_forward_fp8 when no
    gradient is requested): E4M3 H8 [N, D] and W8 [V, D] (torch.uint8) with
    per-tensor scales define the logits; the gradient products use bf16 H, W.
    scale_h / scale_w: Python numbers or CUDA float32 tensors (the device scalar
    at element 0 is read by the kernels)."""
    import torch
    grads = need_dh or need_dw
    if not (H8.is_cuda and W8.is_cuda and labels.is_cuda):
        raise ValueError("H8, W8 and labels must be CUDA tensors")
    if H8.dtype != torch.uint8 or W8.dtype != torch.uint8 or labels.dtype != torch.int32:
        raise TypeError("H8, W8 uint8 (E4M3 bytes), labels int32")
    if not (H8.is_contiguous() and W8.is_contiguous() and labels.is_contiguous()):
        raise ValueError("H8, W8 and labels must be contiguous")
    N, D = H8.shape
    V = W8.shape[0]
    if grads:
        if H is None or W is None:
            raise ValueError("the gradient products need the bf16 H and W")
        _check_inputs(H, W, labels)
    opts = make_options(**options)
    dev = H8.device
    sh = _device_scale(scale_h, dev)
    sw = _device_scale(scale_w, dev)
    out = dict(out or {})
    loss = out.get("loss")
    if loss is None:
        loss = torch.empty(N if options.get("reduction") == "none" else 1, dtype=torch.float32,
                           device=dev)
    lse = out.get("lse")
    if lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    dH = out.get("dH")
    if dH is None and need_dh:
        dH = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
    dW = out.get("dW")
    if dW is None and need_dw:
        dt = torch.float32 if options.get("dw_dtype", "float32") == "float32" else torch.bfloat16
        dW = torch.empty(V, D, dtype=dt, device=dev)
    if workspace is None:
        size = workspace_size if grads else forward_workspace_size
        workspace = torch.empty(size(N, D, V, opts), dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    wsb = workspace.numel() * workspace.element_size()
    if grads:
        rc = lib.flce_forward_backward_fp8(
            _ptr(H8), _ptr(sh), _ptr(W8), _ptr(sw), _ptr(H), _ptr(W), _ptr(labels),
            N, D, V, ctypes.byref(opts), _ptr(loss), _ptr(lse), _ptr(dH) if need_dh else None,
            _ptr(dW) if need_dw else None, _ptr(workspace), wsb, _ptr(status), stream)
    else:
        rc = lib.flce_forward_fp8(_ptr(H8), _ptr(sh), _ptr(W8), _ptr(sw),
                                  _ptr(labels), N, D, V, ctypes.byref(opts), _ptr(loss),
                                  _ptr(lse), _ptr(workspace), wsb, _ptr(status), stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_forward_backward_fp8" if grads else "flce_forward_fp8")
    return Result(loss, lse, dH if need_dh else None, dW if need_dw else None, status)


def scale_grads(dH, dW, scale, stream=None) -> None:
    """dH *= scale and dW *= scale in place (flce_scale_grads); scale is a
    one-element float32 CUDA tensor. Either gradient may be None."""
    import torch
    if scale.dtype != torch.float32 or scale.numel() != 1 or not scale.is_cuda:
        raise TypeError("scale must be a one-element float32 CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream(scale.device).cuda_stream
    dw_dtype = DW_DTYPES["bfloat16" if (dW is not None and dW.dtype == torch.bfloat16) else "float32"]
    rc = lib.flce_scale_grads(_ptr(dH), dH.numel() if dH is not None else 0, _ptr(dW),
                              dW.numel() if dW is not None else 0, dw_dtype, _ptr(scale), stream)
    if rc != FLCE_OK:
        raise FLCEError(rc, "flce_scale_grads")


def check_status(status, stream=None) -> int:
    """Synchronise the stream and return the device status word (0 = ok)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(status.device).cuda_stream
    return int(lib.flce_check_status(_ptr(status), stream))
