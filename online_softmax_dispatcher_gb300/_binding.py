"""ctypes binding of libosd_softmax.so (C ABI: include/softmax.h).

Argument marshalling only: every step of the softmax runs in the library's
CUDA kernels.  The raw functions keep the C names and return the C status
code; out-parameters come back as extra tuple members.  ``softmax`` is the
torch convenience wrapper (torch supplies device memory and the stream).

The library is loaded from the package's in-tree build directory.  If it is
missing the import of any function raises ``SoftmaxLibraryMissing``: there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

F32, F16, BF16 = 0, 1, 2

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED_DTYPE = -2
ERR_ALIAS = -3
ERR_CUDA = -4
ERR_UNSUPPORTED_SHAPE = -5
ERR_DEVICE_TIMEOUT = -6

VARIANT_AUTO = 0
VARIANT_ROWGROUP = 1
VARIANT_BLOCK = 2
VARIANT_BLOCK_TMA = 3
VARIANT_STREAM = 4
VARIANT_SPLITK = 5
VARIANT_SPLITK_WIDE = 6
VARIANT_SPLITK_GRID = 7
VARIANT_COUNT = 8
VARIANTS = {"auto": 0, "rowgroup": 1, "block": 2, "block_tma": 3, "stream": 4, "splitk": 5, "splitk_wide": 6,
            "splitk_grid": 7}

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libosd_softmax.so")

# Exported symbols (kept equal to the declarations in include/softmax.h; a
# host test checks both directions).
EXPORTS = (
    "softmax_fwd", "softmax_fwd_variant", "softmax_fwd_plan", "softmax_query_variant",
    "softmax_plan", "softmax_device_query", "softmax_get_device_error",
    "softmax_last_cuda_error", "softmax_strerror", "softmax_variant_name", "softmax_abi_version",
    "softmax_selftest_bounded_wait", "softmax_bwd", "softmax_bwd_variant", "softmax_fwd_ws",
    "softmax_workspace_size", "softmax_fwd_noalloc", "softmax_fwd_masked", "softmax_fwd_masked_variant",
    "layernorm_fwd", "rmsnorm_fwd", "norm_fwd_variant", "softmax_bwd_plan", "softmax_masked_plan", "norm_plan",
)
LAYERNORM, RMSNORM = 0, 1


class SoftmaxLibraryMissing(RuntimeError):
    pass


class SoftmaxError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = f"softmax: {strerror(status)} (status {status})"
        if status == ERR_CUDA:
            msg += f", cudaError {softmax_last_cuda_error()}"
        super().__init__(msg + (f": {what}" if what else ""))


class DeviceInfo(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int), ("max_smem_optin", ctypes.c_int),
                ("cluster_launch", ctypes.c_int), ("l2_bytes", ctypes.c_int),
                ("cc_major", ctypes.c_int), ("cc_minor", ctypes.c_int)]


class LaunchPlan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("lanes_per_row", ctypes.c_int),
                ("chunks_per_thread", ctypes.c_int), ("rows_per_tile", ctypes.c_int),
                ("stages", ctypes.c_int), ("block_threads", ctypes.c_int),
                ("grid_x", ctypes.c_int64), ("grid_y", ctypes.c_int64), ("cluster_x", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("aligned", ctypes.c_int), ("y_vector", ctypes.c_int),
                ("back_passes", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises SoftmaxLibraryMissing when it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise SoftmaxLibraryMissing(
                    f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
                    "or `python online_softmax_dispatcher_gb300/build.py` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            sig = {
                "softmax_fwd": [vp, vp, i64, i64, i32, vp],
                "softmax_fwd_variant": [vp, vp, i64, i64, i32, i32, vp],
                "softmax_fwd_plan": [vp, vp, i64, i64, i32, ctypes.POINTER(LaunchPlan), vp],
                "softmax_query_variant": [vp, vp, i64, i64, i32, ctypes.POINTER(ctypes.c_int)],
                "softmax_plan": [ctypes.POINTER(DeviceInfo), vp, vp, i64, i64, i32, i32,
                                 ctypes.POINTER(LaunchPlan)],
                "softmax_device_query": [ctypes.POINTER(DeviceInfo)],
                "softmax_get_device_error": [vp, ctypes.POINTER(ctypes.c_uint)],
                "softmax_last_cuda_error": [],
                "softmax_strerror": [i32],
                "softmax_variant_name": [i32],
                "softmax_abi_version": [],
                "softmax_selftest_bounded_wait": [vp, ctypes.c_uint],
                "softmax_bwd": [vp, vp, vp, i64, i64, i32, vp],
                "softmax_bwd_variant": [vp, vp, vp, i64, i64, i32, i32, vp],
                "softmax_fwd_ws": [vp, vp, i64, i64, i32, vp, ctypes.c_uint64, vp],
                "softmax_workspace_size": [vp, vp, i64, i64, i32, ctypes.POINTER(ctypes.c_uint64)],
                "softmax_fwd_noalloc": [vp, vp, i64, i64, i32, vp],
                "softmax_fwd_masked": [vp, vp, i64, i64, i32, ctypes.c_float, vp, i64, i64, vp],
                "softmax_fwd_masked_variant": [vp, vp, i64, i64, i32, ctypes.c_float, vp, i64, i64, i32, vp],
                "layernorm_fwd": [vp, vp, i64, i64, i32, vp, vp, ctypes.c_float, vp, vp, vp],
                "rmsnorm_fwd": [vp, vp, i64, i64, i32, vp, ctypes.c_float, vp, vp],
                "norm_fwd_variant": [i32, vp, vp, i64, i64, i32, vp, vp, ctypes.c_float, vp, vp, i32, vp],
                "softmax_bwd_plan": [ctypes.POINTER(DeviceInfo), vp, vp, vp, i64, i64, i32, i32,
                                     ctypes.POINTER(LaunchPlan)],
                "softmax_masked_plan": [ctypes.POINTER(DeviceInfo), vp, vp, i64, i64, i32, i32,
                                        ctypes.POINTER(LaunchPlan)],
                "norm_plan": [ctypes.POINTER(DeviceInfo), i32, vp, vp, i64, i64, i32, vp, vp, i32,
                              ctypes.POINTER(LaunchPlan)],
            }
            for name, args in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            L.softmax_strerror.restype = ctypes.c_char_p
            L.softmax_variant_name.restype = ctypes.c_char_p
            _lib = L
    return _lib


# ----------------------------------------------------------------------------- raw C entry points


def softmax_fwd(x: int, y: int, rows: int, cols: int, dtype: int, stream: int = 0) -> int:
    return lib().softmax_fwd(x, y, rows, cols, dtype, stream or None)


def softmax_fwd_variant(x: int, y: int, rows: int, cols: int, dtype: int, variant: int,
                        stream: int = 0) -> int:
    return lib().softmax_fwd_variant(x, y, rows, cols, dtype, variant, stream or None)


def softmax_fwd_plan(x: int, y: int, rows: int, cols: int, dtype: int, plan: LaunchPlan,
                     stream: int = 0) -> int:
    return lib().softmax_fwd_plan(x, y, rows, cols, dtype, ctypes.byref(plan), stream or None)


def softmax_fwd_ws(x: int, y: int, rows: int, cols: int, dtype: int, workspace: int, workspace_bytes: int,
                   stream: int = 0) -> int:
    return lib().softmax_fwd_ws(x, y, rows, cols, dtype, workspace or None, workspace_bytes, stream or None)


def softmax_fwd_masked(x: int, y: int, rows: int, cols: int, dtype: int, scale: float, mask: int,
                       mask_rows: int, causal_q: int, stream: int = 0) -> int:
    return lib().softmax_fwd_masked(x, y, rows, cols, dtype, scale, mask or None, mask_rows, causal_q,
                                    stream or None)


def layernorm_fwd(x: int, y: int, rows: int, cols: int, dtype: int, gamma: int, beta: int, eps: float, mean: int,
                  rstd: int, stream: int = 0) -> int:
    return lib().layernorm_fwd(x, y, rows, cols, dtype, gamma or None, beta or None, eps, mean or None,
                               rstd or None, stream or None)


def rmsnorm_fwd(x: int, y: int, rows: int, cols: int, dtype: int, gamma: int, eps: float, rstd: int,
                stream: int = 0) -> int:
    return lib().rmsnorm_fwd(x, y, rows, cols, dtype, gamma or None, eps, rstd or None, stream or None)


def norm_fwd_variant(kind: int, x: int, y: int, rows: int, cols: int, dtype: int, gamma: int, beta: int,
                     eps: float, mean: int, rstd: int, variant: int, stream: int = 0) -> int:
    return lib().norm_fwd_variant(kind, x, y, rows, cols, dtype, gamma or None, beta or None, eps, mean or None,
                                  rstd or None, variant, stream or None)


def softmax_fwd_masked_variant(x: int, y: int, rows: int, cols: int, dtype: int, scale: float, mask: int,
                               mask_rows: int, causal_q: int, variant: int, stream: int = 0) -> int:
    return lib().softmax_fwd_masked_variant(x, y, rows, cols, dtype, scale, mask or None, mask_rows, causal_q,
                                            variant, stream or None)


def softmax_fwd_noalloc(x: int, y: int, rows: int, cols: int, dtype: int, stream: int = 0) -> int:
    return lib().softmax_fwd_noalloc(x, y, rows, cols, dtype, stream or None)


def softmax_workspace_size(x: int, y: int, rows: int, cols: int, dtype: int) -> tuple[int, int]:
    b = ctypes.c_uint64(0)
    rc = lib().softmax_workspace_size(x, y, rows, cols, dtype, ctypes.byref(b))
    return rc, b.value


def softmax_bwd(y: int, dy: int, dx: int, rows: int, cols: int, dtype: int, stream: int = 0) -> int:
    return lib().softmax_bwd(y, dy, dx, rows, cols, dtype, stream or None)


def softmax_bwd_variant(y: int, dy: int, dx: int, rows: int, cols: int, dtype: int, variant: int,
                        stream: int = 0) -> int:
    return lib().softmax_bwd_variant(y, dy, dx, rows, cols, dtype, variant, stream or None)


def softmax_query_variant(x: int, y: int, rows: int, cols: int, dtype: int) -> tuple[int, int]:
    v = ctypes.c_int(-1)
    rc = lib().softmax_query_variant(x, y, rows, cols, dtype, ctypes.byref(v))
    return rc, v.value


def softmax_plan(dev: DeviceInfo, x: int, y: int, rows: int, cols: int, dtype: int,
                 variant: int = VARIANT_AUTO) -> tuple[int, LaunchPlan]:
    p = LaunchPlan()
    rc = lib().softmax_plan(ctypes.byref(dev), x, y, rows, cols, dtype, variant, ctypes.byref(p))
    return rc, p


def softmax_bwd_plan(dev: DeviceInfo, y: int, dy: int, dx: int, rows: int, cols: int, dtype: int,
                     variant: int = VARIANT_AUTO) -> tuple[int, LaunchPlan]:
    p = LaunchPlan()
    rc = lib().softmax_bwd_plan(ctypes.byref(dev), y, dy, dx, rows, cols, dtype, variant, ctypes.byref(p))
    return rc, p


def softmax_masked_plan(dev: DeviceInfo, x: int, y: int, rows: int, cols: int, dtype: int,
                        variant: int = VARIANT_AUTO) -> tuple[int, LaunchPlan]:
    p = LaunchPlan()
    rc = lib().softmax_masked_plan(ctypes.byref(dev), x, y, rows, cols, dtype, variant, ctypes.byref(p))
    return rc, p


def norm_plan(dev: DeviceInfo, kind: int, x: int, y: int, rows: int, cols: int, dtype: int, gamma: int = 0,
              beta: int = 0, variant: int = VARIANT_AUTO) -> tuple[int, LaunchPlan]:
    p = LaunchPlan()
    rc = lib().norm_plan(ctypes.byref(dev), kind, x, y, rows, cols, dtype, gamma or None, beta or None, variant,
                         ctypes.byref(p))
    return rc, p


def softmax_device_query() -> tuple[int, DeviceInfo]:
    d = DeviceInfo()
    rc = lib().softmax_device_query(ctypes.byref(d))
    return rc, d


def softmax_get_device_error(stream: int = 0) -> tuple[int, int]:
    code = ctypes.c_uint(0)
    rc = lib().softmax_get_device_error(stream or None, ctypes.byref(code))
    return rc, code.value


def softmax_selftest_bounded_wait(stream: int = 0, limit_us: int = 20000) -> int:
    return lib().softmax_selftest_bounded_wait(stream or None, limit_us)


def softmax_last_cuda_error() -> int:
    return lib().softmax_last_cuda_error()


def softmax_strerror(status: int) -> str:
    return lib().softmax_strerror(status).decode()


def softmax_variant_name(variant: int) -> str:
    return lib().softmax_variant_name(variant).decode()


def softmax_abi_version() -> int:
    return lib().softmax_abi_version()


def strerror(status: int) -> str:
    try:
        return softmax_strerror(status)
    except SoftmaxLibraryMissing:
        return f"status {status}"


# ----------------------------------------------------------------------------- torch convenience

_TORCH_DTYPES = None


def dtype_code(t_dtype) -> int:
    global _TORCH_DTYPES
    if _TORCH_DTYPES is None:
        import torch

        _TORCH_DTYPES = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
    try:
        return _TORCH_DTYPES[t_dtype]
    except KeyError:
        raise SoftmaxError(ERR_UNSUPPORTED_DTYPE, str(t_dtype)) from None


def softmax(x, *, out=None, variant: int | str = VARIANT_AUTO, plan: LaunchPlan | None = None,
            stream=None, workspace=None):
    """y = softmax(x) over the last dimension of a contiguous CUDA tensor.

    `out` (same shape and dtype, contiguous; x itself for an in-place call,
    else not overlapping x) receives the result when given; `variant` forces a
    kernel; `plan` launches a
    caller-built plan; `stream` is a torch.cuda.Stream (default: current);
    `workspace` (a CUDA tensor of at least softmax_workspace_size bytes) lets
    few, very long rows use every SM (softmax_fwd_ws).
    """
    import torch

    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise SoftmaxError(ERR_INVALID_ARG, "x must be a CUDA tensor")
    if not x.is_contiguous():
        raise SoftmaxError(ERR_INVALID_ARG, "x must be contiguous")
    if x.dim() == 0:
        raise SoftmaxError(ERR_INVALID_ARG, "x must have at least one dimension")
    dt = dtype_code(x.dtype)
    y = torch.empty_like(x) if out is None else out
    if y.shape != x.shape or y.dtype != x.dtype or not y.is_contiguous() or y.device != x.device:
        raise SoftmaxError(ERR_INVALID_ARG, "out must match x in shape, dtype and device and be contiguous")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    if isinstance(variant, str):
        variant = VARIANTS[variant]
    with torch.cuda.device(x.device):
        if workspace is not None:
            if plan is not None or variant != VARIANT_AUTO:
                raise SoftmaxError(ERR_INVALID_ARG, "workspace goes with the dispatcher's choice only")
            rc = softmax_fwd_ws(x.data_ptr(), y.data_ptr(), rows, cols, dt, workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), s)
        elif plan is not None:
            rc = softmax_fwd_plan(x.data_ptr(), y.data_ptr(), rows, cols, dt, plan, s)
        else:
            rc = softmax_fwd_variant(x.data_ptr(), y.data_ptr(), rows, cols, dt, variant, s)
    if rc != OK:
        raise SoftmaxError(rc)
    return y


def softmax_(x, **kw):
    """In-place softmax over the last dimension: x is overwritten with softmax(x)."""
    return softmax(x, out=x, **kw)


def softmax_masked(x, *, scale: float = 1.0, mask=None, causal: bool = False, out=None,
                   variant: int | str = VARIANT_AUTO, stream=None):
    """softmax(scale * x + mask) over the last dimension with an optional causal
    cut, for contiguous CUDA attention scores x of shape [..., Sq, Sk].  mask
    (same dtype) broadcasts over the leading dimensions: [Sk], [1, Sk] or
    [Sq, Sk]; causal=True cuts keys j > i + (Sk - Sq) for query i."""
    import torch

    if not isinstance(x, torch.Tensor) or not x.is_cuda or not x.is_contiguous() or x.dim() == 0:
        raise SoftmaxError(ERR_INVALID_ARG, "x must be a contiguous CUDA tensor")
    dt = dtype_code(x.dtype)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    mptr, mrows = 0, 0
    if mask is not None:
        if mask.dtype != x.dtype or not mask.is_cuda or not mask.is_contiguous() or mask.shape[-1] != cols:
            raise SoftmaxError(ERR_INVALID_ARG, "mask must be a contiguous CUDA tensor [..., Sk] of x's dtype")
        mptr, mrows = mask.data_ptr(), mask.numel() // cols
    causal_q = (x.shape[-2] if x.dim() >= 2 else 1) if causal else 0
    y = torch.empty_like(x) if out is None else out
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    if isinstance(variant, str):
        variant = VARIANTS[variant]
    with torch.cuda.device(x.device):
        rc = softmax_fwd_masked_variant(x.data_ptr(), y.data_ptr(), rows, cols, dt, float(scale), mptr, mrows,
                                        causal_q, variant, s)
    if rc != OK:
        raise SoftmaxError(rc)
    return y


def _norm(kind, x, weight, bias, eps, out, mean, rstd, variant, stream):
    import torch

    if not isinstance(x, torch.Tensor) or not x.is_cuda or not x.is_contiguous() or x.dim() == 0:
        raise SoftmaxError(ERR_INVALID_ARG, "x must be a contiguous CUDA tensor")
    dt = dtype_code(x.dtype)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    for name, v in (("weight", weight), ("bias", bias)):
        if v is not None and (v.dtype != x.dtype or not v.is_cuda or not v.is_contiguous() or v.numel() != cols):
            raise SoftmaxError(ERR_INVALID_ARG, f"{name} must be a contiguous CUDA tensor of {cols} x-dtype values")
    for name, v in (("mean", mean), ("rstd", rstd)):
        if v is not None and (v.dtype != torch.float32 or not v.is_cuda or not v.is_contiguous() or v.numel() != rows):
            raise SoftmaxError(ERR_INVALID_ARG, f"{name} must be a contiguous CUDA float32 tensor of {rows} values")
    y = torch.empty_like(x) if out is None else out
    if y.shape != x.shape or y.dtype != x.dtype or not y.is_contiguous() or y.device != x.device:
        raise SoftmaxError(ERR_INVALID_ARG, "out must match x in shape, dtype and device and be contiguous")
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    if isinstance(variant, str):
        variant = VARIANTS[variant]
    ptr = (lambda t: t.data_ptr() if t is not None else 0)
    with torch.cuda.device(x.device):
        rc = norm_fwd_variant(kind, x.data_ptr(), y.data_ptr(), rows, cols, dt, ptr(weight), ptr(bias), float(eps),
                              ptr(mean), ptr(rstd), variant, s)
    if rc != OK:
        raise SoftmaxError(rc)
    return y


def layer_norm(x, weight=None, bias=None, *, eps: float = 1e-5, out=None, mean=None, rstd=None,
               variant: int | str = VARIANT_AUTO, stream=None):
    """LayerNorm over the last dimension of a contiguous CUDA tensor (weight /
    bias: [cols] of x's dtype or None; mean / rstd: optional float32 [rows]
    outputs).  `out` may be x itself (in place)."""
    return _norm(LAYERNORM, x, weight, bias, eps, out, mean, rstd, variant, stream)


def rms_norm(x, weight=None, *, eps: float = 1e-6, out=None, rstd=None, variant: int | str = VARIANT_AUTO,
             stream=None):
    """RMSNorm over the last dimension of a contiguous CUDA tensor."""
    return _norm(RMSNORM, x, weight, None, eps, out, None, rstd, variant, stream)


def softmax_backward(y, dy, *, out=None, variant: int | str = VARIANT_AUTO, stream=None):
    """dx = y * (dy - sum(dy * y, -1)) for contiguous CUDA tensors y (a softmax
    output) and dy (its upstream gradient).  `out` may be dy or y itself (in
    place)."""
    import torch

    for name, t in (("y", y), ("dy", dy)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise SoftmaxError(ERR_INVALID_ARG, f"{name} must be a contiguous CUDA tensor")
    if dy.shape != y.shape or dy.dtype != y.dtype or dy.device != y.device or y.dim() == 0:
        raise SoftmaxError(ERR_INVALID_ARG, "y and dy must match in shape, dtype and device")
    dt = dtype_code(y.dtype)
    dx = torch.empty_like(y) if out is None else out
    if dx.shape != y.shape or dx.dtype != y.dtype or not dx.is_contiguous() or dx.device != y.device:
        raise SoftmaxError(ERR_INVALID_ARG, "out must match y in shape, dtype and device and be contiguous")
    cols = y.shape[-1]
    rows = y.numel() // cols if cols else 0
    s = (stream or torch.cuda.current_stream(y.device)).cuda_stream
    if isinstance(variant, str):
        variant = VARIANTS[variant]
    with torch.cuda.device(y.device):
        rc = softmax_bwd_variant(y.data_ptr(), dy.data_ptr(), dx.data_ptr(), rows, cols, dt, variant, s)
    if rc != OK:
        raise SoftmaxError(rc)
    return dx


def plan_for(x, y, variant: int | str = VARIANT_AUTO) -> LaunchPlan:
    """The plan the dispatcher picks for tensors x -> y on the current device."""
    if isinstance(variant, str):
        variant = VARIANTS[variant]
    rc, dev = softmax_device_query()
    if rc != OK:
        raise SoftmaxError(rc)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    rc, p = softmax_plan(dev, x.data_ptr(), y.data_ptr(), rows, cols, dtype_code(x.dtype), variant)
    if rc != OK:
        raise SoftmaxError(rc)
    return p
