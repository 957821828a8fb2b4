"""GB300 (sm_103a) fused linear cross-entropy.

A thin Python binding over the C ABI in ``include/flce.h`` (``libflce.so``, built
in-tree by ``build.py``). The functions ``flce_forward``, ``flce_backward``,
``flce_workspace_size``, ``flce_check_device_error`` and ``flce_status_string``
marshal torch tensors into pointers and sizes and call the library; every step of
the computation runs in the library's CUDA kernels. There is no CPU fallback: if
the library is missing, ``load_library`` raises.

``linear_cross_entropy`` wraps the two calls in a ``torch.autograd.Function``. W is
[D, V] by default; ``weight_layout="vd"`` takes the [V, D] weight of an
``nn.Linear(D, V, bias=False)`` language-model head as it is (dW then has that layout too).
X and W are bf16, or both f16 (``input_dtype="f16"`` in the options of the ``_ex`` calls;
the autograd wrapper picks it from the tensors).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "FLCEError", "load_library", "library_path", "flce_workspace_size", "flce_forward", "flce_backward",
    "flce_check_device_error", "flce_status_string", "flce_version", "linear_cross_entropy",
    "LinearCrossEntropyFunction", "REDUCTIONS", "STATUS", "logits_bytes", "EXPORTED_SYMBOLS", "FlceOptions",
    "make_options", "flce_forward_ex", "flce_backward_ex", "flce_forward_backward", "flce_shard_stats",
    "flce_combine_shards", "WEIGHT_LAYOUTS", "INPUT_DTYPES", "flce_last_error_detail", "flce_kernel_launches",
    "flce_selftest_wait_timeout", "flce_backward_band_width", "FusedLinearCrossEntropyLoss", "flce_profile_gemms",
    "flce_profile_read", "GEMM_KINDS", "WORKSPACE_KINDS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}
WEIGHT_LAYOUTS = {"dv": 0, "vd": 1}  # flce_weight_layout: W [D, V] or W [V, D]
INPUT_DTYPES = {"bf16": 0, "f16": 1}  # flce_input_dtype of X, W and dX
STATUS = {
    0: "FLCE_OK", 1: "FLCE_ERR_INVALID_ARG", 2: "FLCE_ERR_ALIGNMENT", 3: "FLCE_ERR_UNSUPPORTED_DEVICE",
    4: "FLCE_ERR_WORKSPACE_TOO_SMALL", 5: "FLCE_ERR_REDUCTION_NONE_GRAD", 6: "FLCE_ERR_CUDA",
    7: "FLCE_ERR_BAD_TARGET", 8: "FLCE_ERR_TIMEOUT", 9: "FLCE_ERR_TOO_LARGE", 10: "FLCE_ERR_F16_RANGE",
}
EXPORTED_SYMBOLS = ("flce_workspace_size", "flce_forward", "flce_backward", "flce_check_device_error",
                    "flce_status_string", "flce_version", "flce_forward_noalloc", "flce_forward_ex",
                    "flce_backward_ex", "flce_forward_backward", "flce_shard_stats", "flce_combine_shards",
                    "flce_last_error_detail", "flce_shard_stats_ex", "flce_kernel_launches",
                    "flce_selftest_wait_timeout", "flce_backward_band_width", "flce_profile_gemms",
                    "flce_profile_read")
GEMM_KINDS = ("forward", "gradient", "dW", "dX")  # the order of flce_profile_read's arrays


class FlceOptions(ctypes.Structure):
    """Mirror of ``flce_options`` in include/flce.h."""

    _fields_ = [("softcap", ctypes.c_float), ("bias", ctypes.c_void_p), ("class_weight", ctypes.c_void_p),
                ("predicted", ctypes.c_void_p), ("accuracy", ctypes.c_void_p), ("dbias", ctypes.c_void_p),
                ("dX_f32", ctypes.c_void_p), ("v_offset", ctypes.c_int64), ("v_total", ctypes.c_int64),
                ("row_band", ctypes.c_int64), ("weight_layout", ctypes.c_int32), ("input_dtype", ctypes.c_int32),
                ("accumulate_grads", ctypes.c_int32)]


def _layout(weight_layout) -> int:
    return WEIGHT_LAYOUTS[weight_layout] if isinstance(weight_layout, str) else int(weight_layout)


def _dtype_code(input_dtype) -> int:
    if isinstance(input_dtype, torch.dtype):
        return {torch.bfloat16: 0, torch.float16: 1}[input_dtype]
    return INPUT_DTYPES[input_dtype] if isinstance(input_dtype, str) else int(input_dtype)


def make_options(softcap: float = 0.0, bias=None, class_weight=None, predicted=None, accuracy=None, dbias=None,
                 dX_f32=None, v_offset: int = 0, v_total: int = 0, row_band: int = 0, weight_layout="dv",
                 input_dtype="bf16", accumulate_grads: bool = False):
    """An ``flce_options`` value (device tensors become pointers)."""
    return FlceOptions(float(softcap), _ptr(bias), _ptr(class_weight), _ptr(predicted), _ptr(accuracy),
                       _ptr(dbias), _ptr(dX_f32), int(v_offset), int(v_total), int(row_band),
                       _layout(weight_layout), _dtype_code(input_dtype), 1 if accumulate_grads else 0)


def _check_dtype(X, options) -> None:
    """The options must name X's element type (the library cannot see it)."""
    if not isinstance(X, torch.Tensor):
        return
    want = 1 if X.dtype == torch.float16 else 0
    have = options.input_dtype if options is not None else 0
    if want != have:
        raise TypeError(f"X is {X.dtype} but the options say input_dtype={have}: "
                        "pass make_options(input_dtype=X.dtype)")


def _vocab(W, options) -> int:
    """V from W's shape: [D, V], or [V, D] when the options say so."""
    return W.shape[0] if options is not None and options.weight_layout == 1 else W.shape[1]


class FLCEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        detail = f" ({flce_last_error_detail()})" if status == 6 else ""
        super().__init__(f"{where}: {flce_status_string(status)}{detail}")


def library_path() -> str:
    return os.path.join(_HERE, "libflce.so")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libflce.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with `python -m linear_cross_entropy_tcgen05_gb300.build`")
    lib = ctypes.CDLL(p)
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.flce_workspace_size.argtypes = [i64, i64, i64, ctypes.c_int]
    lib.flce_workspace_size.restype = sz
    lib.flce_forward.argtypes = [vp, vp, vp, i64, i64, i64, i32, f32, f32, ctypes.c_int, vp, vp, vp, sz, vp]
    lib.flce_forward.restype = ctypes.c_int
    lib.flce_backward.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, f32, f32, ctypes.c_int, vp, vp, vp, vp,
                                  sz, vp]
    lib.flce_backward.restype = ctypes.c_int
    lib.flce_check_device_error.argtypes = [vp, vp]
    lib.flce_check_device_error.restype = ctypes.c_int
    lib.flce_status_string.argtypes = [ctypes.c_int]
    lib.flce_status_string.restype = ctypes.c_char_p
    lib.flce_version.argtypes = []
    lib.flce_version.restype = ctypes.c_int
    lib.flce_last_error_detail.argtypes = []
    lib.flce_last_error_detail.restype = ctypes.c_char_p
    lib.flce_kernel_launches.argtypes = []
    lib.flce_kernel_launches.restype = ctypes.c_ulonglong
    lib.flce_selftest_wait_timeout.argtypes = [vp, sz, vp]
    lib.flce_selftest_wait_timeout.restype = ctypes.c_int
    lib.flce_backward_band_width.argtypes = [i64, i64, i64, vp]
    lib.flce_backward_band_width.restype = i64
    lib.flce_profile_gemms.argtypes = [ctypes.c_int]
    lib.flce_profile_gemms.restype = None
    lib.flce_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_ulonglong)]
    lib.flce_profile_read.restype = ctypes.c_int
    op = ctypes.POINTER(FlceOptions)
    lib.flce_forward_ex.argtypes = [vp, vp, vp, i64, i64, i64, i32, f32, f32, ctypes.c_int, op, vp, vp, vp, sz, vp]
    lib.flce_forward_ex.restype = ctypes.c_int
    lib.flce_backward_ex.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, f32, f32, ctypes.c_int, op, vp, vp, vp,
                                     vp, sz, vp]
    lib.flce_backward_ex.restype = ctypes.c_int
    lib.flce_forward_backward.argtypes = [vp, vp, vp, i64, i64, i64, i32, f32, f32, ctypes.c_int, op, vp, vp, vp,
                                          vp, vp, vp, sz, vp]
    lib.flce_forward_backward.restype = ctypes.c_int
    lib.flce_shard_stats.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, vp, vp, sz, vp]
    lib.flce_shard_stats.restype = ctypes.c_int
    lib.flce_shard_stats_ex.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, vp, vp, vp, sz, vp]
    lib.flce_shard_stats_ex.restype = ctypes.c_int
    lib.flce_combine_shards.argtypes = [vp, i32, vp, i64, i64, i32, f32, f32, ctypes.c_int, vp, vp, vp, sz, vp]
    lib.flce_combine_shards.restype = ctypes.c_int
    if path is None:
        _LIB = lib
    return lib


def flce_status_string(status: int) -> str:
    return load_library().flce_status_string(int(status)).decode()


def flce_version() -> int:
    return int(load_library().flce_version())


def flce_selftest_wait_timeout(workspace, stream=None) -> int:
    """Launch the bounded-wait self-test (returns the launch status; read the outcome
    with flce_check_device_error, which should give FLCE_ERR_TIMEOUT after ~2 s)."""
    return int(load_library().flce_selftest_wait_timeout(_ptr(workspace), _nbytes(workspace), _stream(stream)))


def flce_backward_band_width(N: int, D: int, V: int, options: FlceOptions | None = None) -> int:
    """Vocabulary columns per gradient band that flce_backward uses on this device (0 if none)."""
    return int(load_library().flce_backward_band_width(N, D, V, _opt_ref(options)))


def flce_kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load_library().flce_kernel_launches())


def flce_profile_gemms(enable: bool) -> None:
    """Bracket every later GEMM launch with CUDA events (diagnostics), or stop."""
    load_library().flce_profile_gemms(1 if enable else 0)


def flce_profile_read() -> dict:
    """{kind: (device ms summed, launches)} of the GEMM launches timed since the last read
    (kinds as in GEMM_KINDS); waits for their events."""
    ms = (ctypes.c_double * 4)()
    n = (ctypes.c_ulonglong * 4)()
    _check(load_library().flce_profile_read(ms, n), "flce_profile_read")
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(GEMM_KINDS)}


def flce_last_error_detail() -> str:
    """The CUDA call behind the calling thread's last FLCE_ERR_CUDA ('' if none)."""
    return load_library().flce_last_error_detail().decode()


WORKSPACE_KINDS = {"forward": 0, "backward": 1, "both": 2, "forward_valid_rows": 3}


def flce_workspace_size(N: int, D: int, V: int, for_backward) -> int:
    """Workspace bytes: for_backward False/True (forward / backward), or one of
    WORKSPACE_KINDS by name or number ("forward_valid_rows": the size from which the
    forward runs its GEMM on the valid rows only)."""
    if isinstance(for_backward, str):
        which = WORKSPACE_KINDS[for_backward]
    elif isinstance(for_backward, bool):
        which = 1 if for_backward else 0
    else:
        which = int(for_backward)
    return int(load_library().flce_workspace_size(N, D, V, which))


def logits_bytes(N: int, V: int, elem_bytes: int) -> int:
    """Bytes of an N x V logits buffer (what the fused path never allocates)."""
    return int(N) * int(V) * int(elem_bytes)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr() if isinstance(t, torch.Tensor) else int(t)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str) -> None:
    if status != 0:
        raise FLCEError(status, where)


def _nbytes(t) -> int:
    return t.numel() * t.element_size() if isinstance(t, torch.Tensor) else 0


def flce_forward(X, W, targets, loss, lse, workspace, ignore_index: int = -100, label_smoothing: float = 0.0,
                 zloss_scale: float = 0.0, reduction: str = "mean", stream=None, N=None, D=None, V=None,
                 ws_bytes=None, raise_on_error: bool = True) -> int:
    """Call flce_forward. Tensors are device tensors laid out as in flce.h; returns the status."""
    _check_dtype(X, None)
    N = X.shape[0] if N is None else N
    D = X.shape[1] if D is None else D
    V = W.shape[1] if V is None else V
    st = load_library().flce_forward(
        _ptr(X), _ptr(W), _ptr(targets), N, D, V, int(ignore_index), float(label_smoothing), float(zloss_scale),
        REDUCTIONS[reduction] if isinstance(reduction, str) else int(reduction), _ptr(loss), _ptr(lse),
        _ptr(workspace), _nbytes(workspace) if ws_bytes is None else int(ws_bytes), _stream(stream))
    if raise_on_error:
        _check(st, "flce_forward")
    return st


def flce_backward(X, W, targets, lse, grad_out, dX, dW, workspace, ignore_index: int = -100,
                  label_smoothing: float = 0.0, zloss_scale: float = 0.0, reduction: str = "mean", stream=None,
                  N=None, D=None, V=None, ws_bytes=None, raise_on_error: bool = True) -> int:
    """Call flce_backward (grad_out is a device fp32 scalar tensor); returns the status."""
    _check_dtype(X, None)
    N = X.shape[0] if N is None else N
    D = X.shape[1] if D is None else D
    V = W.shape[1] if V is None else V
    st = load_library().flce_backward(
        _ptr(X), _ptr(W), _ptr(targets), _ptr(lse), N, D, V, int(ignore_index), float(label_smoothing),
        float(zloss_scale), REDUCTIONS[reduction] if isinstance(reduction, str) else int(reduction),
        _ptr(grad_out), _ptr(dX), _ptr(dW), _ptr(workspace),
        _nbytes(workspace) if ws_bytes is None else int(ws_bytes), _stream(stream))
    if raise_on_error:
        _check(st, "flce_backward")
    return st


def _red(reduction) -> int:
    return REDUCTIONS[reduction] if isinstance(reduction, str) else int(reduction)


def _opt_ref(options):
    return ctypes.byref(options) if options is not None else None


def flce_forward_ex(X, W, targets, loss, lse, workspace, ignore_index: int = -100, label_smoothing: float = 0.0,
                    zloss_scale: float = 0.0, reduction: str = "mean", options: FlceOptions | None = None,
                    stream=None, raise_on_error: bool = True) -> int:
    """Call flce_forward_ex (``options`` from ``make_options``)."""
    _check_dtype(X, options)
    st = load_library().flce_forward_ex(
        _ptr(X), _ptr(W), _ptr(targets), X.shape[0], X.shape[1], _vocab(W, options), int(ignore_index),
        float(label_smoothing), float(zloss_scale), _red(reduction), _opt_ref(options), _ptr(loss), _ptr(lse),
        _ptr(workspace), _nbytes(workspace), _stream(stream))
    if raise_on_error:
        _check(st, "flce_forward_ex")
    return st


def flce_backward_ex(X, W, targets, lse, grad_out, dX, dW, workspace, ignore_index: int = -100,
                     label_smoothing: float = 0.0, zloss_scale: float = 0.0, reduction: str = "mean",
                     options: FlceOptions | None = None, stream=None, raise_on_error: bool = True) -> int:
    """Call flce_backward_ex (dX may be None when options.dX_f32 is set)."""
    _check_dtype(X, options)
    st = load_library().flce_backward_ex(
        _ptr(X), _ptr(W), _ptr(targets), _ptr(lse), X.shape[0], X.shape[1], _vocab(W, options), int(ignore_index),
        float(label_smoothing), float(zloss_scale), _red(reduction), _opt_ref(options), _ptr(grad_out), _ptr(dX),
        _ptr(dW), _ptr(workspace), _nbytes(workspace), _stream(stream))
    if raise_on_error:
        _check(st, "flce_backward_ex")
    return st


def flce_forward_backward(X, W, targets, grad_out, loss, lse, dX, dW, workspace, ignore_index: int = -100,
                          label_smoothing: float = 0.0, zloss_scale: float = 0.0, reduction: str = "mean",
                          options: FlceOptions | None = None, stream=None, raise_on_error: bool = True) -> int:
    """Call flce_forward_backward (workspace: flce_workspace_size(N, D, V, 2) bytes)."""
    _check_dtype(X, options)
    st = load_library().flce_forward_backward(
        _ptr(X), _ptr(W), _ptr(targets), X.shape[0], X.shape[1], _vocab(W, options), int(ignore_index),
        float(label_smoothing), float(zloss_scale), _red(reduction), _opt_ref(options), _ptr(grad_out), _ptr(loss),
        _ptr(lse), _ptr(dX), _ptr(dW), _ptr(workspace), _nbytes(workspace), _stream(stream))
    if raise_on_error:
        _check(st, "flce_forward_backward")
    return st


def flce_shard_stats(X, W_shard, targets, v_offset: int, stats, workspace, ignore_index: int = -100, stream=None,
                     raise_on_error: bool = True, options: FlceOptions | None = None) -> int:
    """Call flce_shard_stats (or flce_shard_stats_ex with ``options``: weight layout and
    input dtype only): stats is a device fp32 [4, N] tensor."""
    _check_dtype(X, options)
    args = (_ptr(X), _ptr(W_shard), _ptr(targets), X.shape[0], X.shape[1], _vocab(W_shard, options), int(v_offset),
            int(ignore_index))
    tail = (_ptr(stats), _ptr(workspace), _nbytes(workspace), _stream(stream))
    if options is None:
        st = load_library().flce_shard_stats(*args, *tail)
    else:
        st = load_library().flce_shard_stats_ex(*args, ctypes.byref(options), *tail)
    if raise_on_error:
        _check(st, "flce_shard_stats")
    return st


def flce_combine_shards(stats, targets, v_total: int, loss, lse, workspace, ignore_index: int = -100,
                        label_smoothing: float = 0.0, zloss_scale: float = 0.0, reduction: str = "mean",
                        stream=None, raise_on_error: bool = True) -> int:
    """Call flce_combine_shards: stats is a device fp32 [K, 4, N] tensor."""
    st = load_library().flce_combine_shards(
        _ptr(stats), int(stats.shape[0]), _ptr(targets), int(stats.shape[2]), int(v_total), int(ignore_index),
        float(label_smoothing), float(zloss_scale), _red(reduction), _ptr(loss), _ptr(lse), _ptr(workspace),
        _nbytes(workspace), _stream(stream))
    if raise_on_error:
        _check(st, "flce_combine_shards")
    return st


def flce_check_device_error(workspace, stream=None) -> int:
    """Synchronise and read/clear the device error word; returns the status code."""
    return int(load_library().flce_check_device_error(_ptr(workspace), _stream(stream)))


def _workspace(N, D, V, device, for_backward, cache=None):
    need = flce_workspace_size(N, D, V, for_backward)
    if cache is not None and cache.numel() >= need:
        return cache
    return torch.empty(max(need, 16), dtype=torch.uint8, device=device)


def _validate(X, W, targets, layout=0):
    if X.dtype not in (torch.bfloat16, torch.float16) or W.dtype != X.dtype:
        raise TypeError("X and W must both be bfloat16 or both float16")
    if targets.dtype != torch.int32:
        raise TypeError("targets must be int32")
    wd = W.shape[1] if layout == 1 else W.shape[0]
    if X.dim() != 2 or W.dim() != 2 or targets.dim() != 1 or X.shape[1] != wd or X.shape[0] != targets.shape[0]:
        raise ValueError(("expected X [N,D], W [V,D]" if layout == 1 else "expected X [N,D], W [D,V]")
                         + ", targets [N]")
    if not (X.is_cuda and W.is_cuda and targets.is_cuda):
        raise ValueError("X, W and targets must be CUDA tensors")
    if not (W.device == X.device and targets.device == X.device):
        raise ValueError("X, W and targets must be on the same device")
    if not (X.is_contiguous() and W.is_contiguous() and targets.is_contiguous()):
        raise ValueError("X, W and targets must be contiguous")


class LinearCrossEntropyFunction(torch.autograd.Function):
    """loss = CE(softmax(X @ W), targets) with fused tensor-core kernels (no N x V logits)."""

    @staticmethod
    def forward(ctx, X, W, targets, ignore_index=-100, label_smoothing=0.0, zloss_scale=0.0, reduction="mean",
                softcap=0.0, bias=None, class_weight=None, weight_layout="dv", metrics=None):
        layout = _layout(weight_layout)
        _validate(X, W, targets, layout)
        # the library works on the current device and the current stream: make them X's
        with torch.cuda.device(X.device):
            N, D = X.shape
            V = W.shape[0] if layout == 1 else W.shape[1]
            # training: a workspace with room for the valid-row forward (the backward's own
            # workspace, allocated next, is larger, so the peak does not grow); inference: the
            # forward's minimum
            training = bool(ctx.needs_input_grad[0] or ctx.needs_input_grad[1])
            ws = _workspace(N, D, V, X.device, "forward_valid_rows" if training else False)
            loss = torch.empty(N if reduction == "none" else 1, dtype=torch.float32, device=X.device)
            lse = torch.empty(N, dtype=torch.float32, device=X.device)
            b32 = bias.detach().float().contiguous() if bias is not None else None
            w32 = class_weight.detach().float().contiguous() if class_weight is not None else None
            pred = acc = None
            if metrics is not None:  # argmax per row and token accuracy, from the same forward pass
                pred = torch.empty(N, dtype=torch.int32, device=X.device)
                acc = torch.empty(1, dtype=torch.float32, device=X.device)
                metrics["predicted"], metrics["accuracy"] = pred, acc
            opts = make_options(softcap=softcap, bias=b32, class_weight=w32, weight_layout=layout,
                                input_dtype=X.dtype, predicted=pred, accuracy=acc)
            flce_forward_ex(X, W, targets, loss, lse, ws, ignore_index, label_smoothing, zloss_scale, reduction,
                            opts)
            ctx.save_for_backward(X, W, targets, lse)
            ctx.extra = (b32, w32, bias is not None and bias.requires_grad,
                         bias.dtype if bias is not None else None)
            ctx.opts = (ignore_index, label_smoothing, zloss_scale, reduction, softcap, layout)
            return loss if reduction == "none" else loss[0]

    @staticmethod
    def backward(ctx, grad_loss):
        X, W, targets, lse = ctx.saved_tensors
        with torch.cuda.device(X.device):
            b32, w32, want_db, b_dtype = ctx.extra
            ignore_index, label_smoothing, zloss_scale, reduction, softcap, layout = ctx.opts
            if reduction == "none":
                raise RuntimeError("reduction='none' has no fused backward (FLCE_ERR_REDUCTION_NONE_GRAD)")
            N, D = X.shape
            V = W.shape[0] if layout == 1 else W.shape[1]
            ws = _workspace(N, D, V, X.device, True)
            g = grad_loss.detach().to(device=X.device, dtype=torch.float32).reshape(1).contiguous()
            dX = torch.empty_like(X)
            dW = torch.empty(W.shape, dtype=torch.float32, device=X.device)
            db = torch.empty(V, dtype=torch.float32, device=X.device) if want_db else None
            opts = make_options(softcap=softcap, bias=b32, class_weight=w32, dbias=db, weight_layout=layout,
                                input_dtype=X.dtype)
            flce_backward_ex(X, W, targets, lse, g, dX, dW, ws, ignore_index, label_smoothing, zloss_scale,
                             reduction, opts)
            return (dX, dW.to(W.dtype), None, None, None, None, None, None,
                    db.to(b_dtype) if db is not None else None, None, None, None)


def linear_cross_entropy(X, W, targets, ignore_index: int = -100, label_smoothing: float = 0.0,
                         zloss_scale: float = 0.0, reduction: str = "mean", softcap: float = 0.0, bias=None,
                         class_weight=None, weight_layout: str = "dv"):
    """Fused linear cross-entropy of X [N,D], W [D,V] (both bf16 or both f16), int32 targets [N].

    ``weight_layout="vd"`` takes W as [V,D] (an ``nn.Linear(D, V)`` weight) instead.

    Optional: a logit ``softcap``, a ``bias`` [V] (its gradient is returned through
    autograd) and per-class weights ``class_weight`` [V]. The gradient of W is
    accumulated in fp32 by the kernels and returned in W's dtype through autograd; call
    ``flce_backward`` directly to keep the fp32 dW.
    """
    return LinearCrossEntropyFunction.apply(X, W, targets, ignore_index, label_smoothing, zloss_scale, reduction,
                                            softcap, bias, class_weight, weight_layout)


class FusedLinearCrossEntropyLoss(torch.nn.Module):
    """The loss of a language-model head as a module: ``loss(weight, hidden, target,
    bias=None)`` with ``weight`` the [V, D] weight of an ``nn.Linear(D, V)`` head, ``hidden``
    [BT, D] hidden states (bf16 or f16, like the weight) and ``target`` [BT] token ids.

    The options follow the feature list of Liger-Kernel PR #1291 ("Summary"): ``ce_weight``
    (per-class weights), ``ignore_index``, ``lse_square_scale`` (z-loss), ``label_smoothing``,
    ``reduction`` ('mean', 'sum', or 'none' for a forward without gradient), ``softcap``,
    ``return_token_accuracy`` and ``return_predicted_tokens``. With either return flag the
    module returns a tuple (loss, accuracy or None, predicted or None); the extra outputs
    carry no gradient. Targets of any integer type are accepted (converted to int32).
    """

    def __init__(self, ce_weight=None, ignore_index: int = -100, lse_square_scale: float = 0.0,
                 label_smoothing: float = 0.0, reduction: str = "mean", softcap: float | None = None,
                 return_token_accuracy: bool = False, return_predicted_tokens: bool = False):
        super().__init__()
        if reduction not in REDUCTIONS:
            raise ValueError(f"reduction must be one of {sorted(REDUCTIONS)}")
        self.ce_weight = ce_weight
        self.ignore_index = int(ignore_index)
        self.lse_square_scale = float(lse_square_scale)
        self.label_smoothing = float(label_smoothing)
        self.reduction = reduction
        self.softcap = float(softcap or 0.0)
        self.return_token_accuracy = bool(return_token_accuracy)
        self.return_predicted_tokens = bool(return_predicted_tokens)

    def forward(self, weight, hidden, target, bias=None):
        metrics = {} if (self.return_token_accuracy or self.return_predicted_tokens) else None
        loss = LinearCrossEntropyFunction.apply(
            hidden, weight, target.to(torch.int32).contiguous(), self.ignore_index, self.label_smoothing,
            self.lse_square_scale, self.reduction, self.softcap, bias, self.ce_weight, "vd", metrics)
        if metrics is None:
            return loss
        acc = metrics["accuracy"][0] if self.return_token_accuracy else None
        pred = metrics["predicted"] if self.return_predicted_tokens else None
        return loss, acc, pred
