"""ctypes binding of libqk.so with the same names as the C ABI (include/qk.h).

Argument marshalling only: pointers, sizes, dtype codes and streams are
converted and passed through; the operators themselves run in the CUDA
kernels of libqk.so.  A non-OK status raises QkError.  There is no fallback:
if the library is missing every call raises.

The ``softmax_fwd`` / ``rmsnorm_fwd`` / ``layernorm_fwd`` / ``xent_fwd`` helpers take
and return CUDA tensors (they allocate the outputs with PyTorch and then call
the C entry points).
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "_lib", "libqk.so")

QK_F32, QK_BF16 = 0, 1
QK_OP_SOFTMAX, QK_OP_RMSNORM, QK_OP_XENT = 0, 1, 2
QK_OP_SOFTMAX_BWD, QK_OP_RMSNORM_BWD, QK_OP_XENT_BWD = 3, 4, 5
QK_OP_LAYERNORM = 6
QK_OK = 0
QK_ERR_INVALID_ARG = 1
QK_ERR_UNSUPPORTED = 2
QK_ERR_MISALIGNED = 3
QK_ERR_LAUNCH = 4
QK_ERR_TIMEOUT = 5
QK_ERR_NO_DEVICE = 6

_EXPORTS = (
    "qk_softmax_fwd", "qk_rmsnorm_fwd", "qk_xent_fwd", "qk_status_string",
    "qk_get_device_status", "qk_max_row_elements", "qk_get_plan",
    "qk_set_plan_override", "qk_test_wait_timeout", "qk_softmax_bwd", "qk_rmsnorm_bwd",
    "qk_rmsnorm_bwd_workspace_size", "qk_xent_bwd", "qk_rmsnorm_bwd_noalloc",
    "qk_xent_fwd_ex", "qk_xent_bwd_ex", "qk_layernorm_fwd",
)


class QkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {qk_status_string(status)} (status {status})")


class qk_xent_options(ctypes.Structure):
    _fields_ = [("has_ignore_index", ctypes.c_int32), ("z_loss", ctypes.c_float),
                ("ignore_index", ctypes.c_int64)]


class qk_plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "path", "threads", "row_threads", "vec_per_thread", "cluster", "slots", "chunks",
        "ctas_per_sm", "grid", "smem_bytes")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIBRARY):
    """Load libqk.so (once) and declare its signatures; raises if it is missing."""
    global _lib
    lib = _lib
    if lib is not None:  # every call after the first: no lock
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -m memory_bound_row_rmsnorm_gb300.build)")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        fp = ctypes.POINTER(ctypes.c_float)
        lib.qk_softmax_fwd.argtypes = [vp, vp, i64, i64, i32, vp]
        lib.qk_rmsnorm_fwd.argtypes = [vp, vp, vp, vp, i64, i64, ctypes.c_float, i32, vp]
        lib.qk_xent_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i32, vp]
        lib.qk_status_string.argtypes = [i32]
        lib.qk_status_string.restype = ctypes.c_char_p
        lib.qk_get_device_status.argtypes = [vp]
        lib.qk_max_row_elements.argtypes = [i32, i32]
        lib.qk_max_row_elements.restype = i64
        lib.qk_get_plan.argtypes = [i32, i32, i64, i64, ctypes.POINTER(qk_plan)]
        lib.qk_set_plan_override.argtypes = [i32, i32, ctypes.POINTER(qk_plan)]
        lib.qk_test_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.qk_softmax_bwd.argtypes = [vp, vp, vp, i64, i64, i32, vp]
        lib.qk_rmsnorm_bwd_workspace_size.argtypes = [i64, i64, i32, ctypes.POINTER(ctypes.c_size_t)]
        lib.qk_rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i64, i64, i32, vp]
        lib.qk_xent_bwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, vp]
        lib.qk_rmsnorm_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, vp]
        op = ctypes.POINTER(qk_xent_options)
        lib.qk_xent_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, op, vp]
        lib.qk_xent_bwd_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, op, vp]
        lib.qk_layernorm_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, ctypes.c_float, i32, vp]
        for name in ("qk_softmax_fwd", "qk_rmsnorm_fwd", "qk_xent_fwd", "qk_get_device_status",
                     "qk_get_plan", "qk_set_plan_override", "qk_test_wait_timeout",
                     "qk_softmax_bwd", "qk_rmsnorm_bwd_workspace_size", "qk_rmsnorm_bwd",
                     "qk_xent_bwd", "qk_rmsnorm_bwd_noalloc", "qk_xent_fwd_ex", "qk_xent_bwd_ex",
                     "qk_layernorm_fwd"):
            getattr(lib, name).restype = i32
        del fp
        _lib = lib
        return lib


def _ptr(p) -> int | None:
    """A device pointer from an int, None, or anything with data_ptr()."""
    if p is None:
        return None
    if hasattr(p, "data_ptr"):
        return p.data_ptr()
    return int(p)


def _stream(s) -> int | None:
    """A cudaStream_t from an int, a torch.cuda.Stream, or None (torch's current stream)."""
    if s is None:
        import sys
        torch = sys.modules.get("torch")
        if torch is not None and torch.cuda.is_available() and torch.cuda.is_initialized():
            return torch.cuda.current_stream().cuda_stream or None
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream or None
    return int(s) or None


def _check(st: int, where: str) -> None:
    if st != QK_OK:
        raise QkError(st, where)


# --- the C entry points, same names -----------------------------------------
def qk_softmax_fwd(x, y, M: int, N: int, dtype: int, stream=None) -> None:
    _check(load_library().qk_softmax_fwd(_ptr(x), _ptr(y), M, N, dtype, _stream(stream)),
           "qk_softmax_fwd")


def qk_rmsnorm_fwd(x, w, y, rstd, M: int, N: int, eps: float, dtype: int, stream=None) -> None:
    _check(load_library().qk_rmsnorm_fwd(_ptr(x), _ptr(w), _ptr(y), _ptr(rstd), M, N, eps, dtype,
                                         _stream(stream)), "qk_rmsnorm_fwd")


def qk_layernorm_fwd(x, w, b, y, mean, rstd, M: int, N: int, eps: float, dtype: int,
                     stream=None) -> None:
    _check(load_library().qk_layernorm_fwd(_ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(mean),
                                           _ptr(rstd), M, N, eps, dtype, _stream(stream)),
           "qk_layernorm_fwd")


def qk_xent_fwd(logits, targets, loss, lse, M: int, N: int, dtype: int, stream=None) -> None:
    _check(load_library().qk_xent_fwd(_ptr(logits), _ptr(targets), _ptr(loss), _ptr(lse), M, N,
                                      dtype, _stream(stream)), "qk_xent_fwd")


def qk_softmax_bwd(y, dy, dx, M: int, N: int, dtype: int, stream=None) -> None:
    _check(load_library().qk_softmax_bwd(_ptr(y), _ptr(dy), _ptr(dx), M, N, dtype, _stream(stream)),
           "qk_softmax_bwd")


def qk_rmsnorm_bwd_workspace_size(M: int, N: int, dtype: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().qk_rmsnorm_bwd_workspace_size(M, N, dtype, ctypes.byref(n)),
           "qk_rmsnorm_bwd_workspace_size")
    return n.value


def qk_rmsnorm_bwd(x, w, rstd, dy, dx, dw, workspace, workspace_bytes: int, M: int, N: int,
                   dtype: int, stream=None) -> None:
    _check(load_library().qk_rmsnorm_bwd(_ptr(x), _ptr(w), _ptr(rstd), _ptr(dy), _ptr(dx), _ptr(dw),
                                         _ptr(workspace), int(workspace_bytes), M, N, dtype,
                                         _stream(stream)), "qk_rmsnorm_bwd")


def qk_rmsnorm_bwd_noalloc(x, w, rstd, dy, dx, dw, M: int, N: int, dtype: int, stream=None) -> None:
    """qk_rmsnorm_bwd with the workspace taken from the library's fixed device
    array (for callers that cannot allocate device memory)."""
    _check(load_library().qk_rmsnorm_bwd_noalloc(_ptr(x), _ptr(w), _ptr(rstd), _ptr(dy), _ptr(dx),
                                                 _ptr(dw), M, N, dtype, _stream(stream)),
           "qk_rmsnorm_bwd_noalloc")


def qk_xent_bwd(logits, targets, lse, dloss, dlogits, M: int, N: int, dtype: int, stream=None) -> None:
    _check(load_library().qk_xent_bwd(_ptr(logits), _ptr(targets), _ptr(lse), _ptr(dloss),
                                      _ptr(dlogits), M, N, dtype, _stream(stream)), "qk_xent_bwd")


def _options(ignore_index, z_loss):
    if ignore_index is None and not z_loss:
        return None
    return ctypes.byref(qk_xent_options(
        0 if ignore_index is None else 1, float(z_loss), 0 if ignore_index is None else int(ignore_index)))


def qk_xent_fwd_ex(logits, targets, loss, lse, mean_loss, M: int, N: int, dtype: int,
                   ignore_index=None, z_loss: float = 0.0, stream=None) -> None:
    _check(load_library().qk_xent_fwd_ex(_ptr(logits), _ptr(targets), _ptr(loss), _ptr(lse),
                                         _ptr(mean_loss), M, N, dtype, _options(ignore_index, z_loss),
                                         _stream(stream)), "qk_xent_fwd_ex")


def qk_xent_bwd_ex(logits, targets, lse, dloss, dlogits, M: int, N: int, dtype: int,
                   ignore_index=None, z_loss: float = 0.0, stream=None) -> None:
    _check(load_library().qk_xent_bwd_ex(_ptr(logits), _ptr(targets), _ptr(lse), _ptr(dloss),
                                         _ptr(dlogits), M, N, dtype, _options(ignore_index, z_loss),
                                         _stream(stream)), "qk_xent_bwd_ex")


def qk_status_string(status: int) -> str:
    return load_library().qk_status_string(status).decode()


def qk_get_device_status(stream=None) -> int:
    """Returns (does not raise) the device status word, clearing it."""
    return load_library().qk_get_device_status(_stream(stream))


def qk_max_row_elements(op: int, dtype: int) -> int:
    return load_library().qk_max_row_elements(op, dtype)


def qk_get_plan(op: int, dtype: int, M: int, N: int) -> dict:
    p = qk_plan()
    _check(load_library().qk_get_plan(op, dtype, M, N, ctypes.byref(p)), "qk_get_plan")
    return p.as_dict()


def qk_set_plan_override(op: int, dtype: int, plan: dict | None) -> None:
    if plan is None:
        _check(load_library().qk_set_plan_override(op, dtype, None), "qk_set_plan_override")
        return
    p = qk_plan(**{k: int(v) for k, v in plan.items() if k in dict(qk_plan._fields_)})
    _check(load_library().qk_set_plan_override(op, dtype, ctypes.byref(p)), "qk_set_plan_override")


def qk_test_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(load_library().qk_test_wait_timeout(int(timeout_ns), _stream(stream)),
           "qk_test_wait_timeout")


# --- tensor helpers ----------------------------------------------------------
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return QK_F32
    if t.dtype == torch.bfloat16:
        return QK_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16 expected")


def _rows(x):
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    N = x.shape[-1] if x.dim() > 0 else 1
    return x.numel() // max(N, 1), N


def softmax_fwd(x, out=None, stream=None):
    """Row-wise softmax over the last dimension of a CUDA tensor."""
    import torch
    M, N = _rows(x)
    y = torch.empty_like(x) if out is None else out
    qk_softmax_fwd(x, y, M, N, _dtype_code(x), stream)
    return y


def rmsnorm_fwd(x, w, eps: float = 1e-6, out=None, want_rstd: bool = True, stream=None):
    """RMSNorm over the last dimension; returns (y, rstd) (rstd is None if not wanted)."""
    import torch
    M, N = _rows(x)
    if w.dtype != x.dtype or w.numel() != N or not w.is_contiguous():
        raise ValueError("w must be a contiguous [N] tensor of x's dtype")
    y = torch.empty_like(x) if out is None else out
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if want_rstd else None
    qk_rmsnorm_fwd(x, w, y, rstd, M, N, eps, _dtype_code(x), stream)
    return y, rstd


def layernorm_fwd(x, w, b=None, eps: float = 1e-5, out=None, want_stats: bool = True,
                  stream=None):
    """LayerNorm over the last dimension; returns (y, mean, rstd) (the two
    statistics are None if not wanted).  b may be None (no bias)."""
    import torch
    M, N = _rows(x)
    for name, t in (("w", w), ("b", b)):
        if t is not None and (t.dtype != x.dtype or t.numel() != N or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous [N] tensor of x's dtype")
    y = torch.empty_like(x) if out is None else out
    mean = rstd = None
    if want_stats:
        mean = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    qk_layernorm_fwd(x, w, b, y, mean, rstd, M, N, eps, _dtype_code(x), stream)
    return y, mean, rstd


def xent_fwd(logits, targets, want_lse: bool = True, ignore_index=None, z_loss: float = 0.0,
             want_mean: bool = False, stream=None):
    """Per-row cross-entropy; returns (loss, lse) (lse is None if not wanted),
    or (loss, lse, mean) with want_mean."""
    import torch
    M, N = _rows(logits)
    if targets.dtype != torch.int64 or targets.numel() != M or not targets.is_contiguous():
        raise ValueError("targets must be a contiguous int64 tensor with one entry per row")
    loss = torch.empty(logits.shape[:-1], dtype=torch.float32, device=logits.device)
    lse = torch.empty_like(loss) if want_lse else None
    if ignore_index is None and not z_loss and not want_mean:
        qk_xent_fwd(logits, targets, loss, lse, M, N, _dtype_code(logits), stream)
        return loss, lse
    mean = torch.empty((), dtype=torch.float32, device=logits.device) if want_mean else None
    qk_xent_fwd_ex(logits, targets, loss, lse, mean, M, N, _dtype_code(logits), ignore_index, z_loss,
                   stream)
    return (loss, lse, mean) if want_mean else (loss, lse)


def softmax_bwd(y, dy, out=None, stream=None):
    """Softmax backward over the last dimension: y * (dy - sum(dy * y))."""
    import torch
    M, N = _rows(y)
    dx = torch.empty_like(y) if out is None else out
    qk_softmax_bwd(y, dy, dx, M, N, _dtype_code(y), stream)
    return dx


def rmsnorm_bwd(x, w, rstd, dy, stream=None):
    """RMSNorm backward; returns (dx, dw) with dw in float32.  Allocates the
    workspace with PyTorch (the library itself allocates nothing)."""
    import torch
    M, N = _rows(x)
    code = _dtype_code(x)
    ws_bytes = qk_rmsnorm_bwd_workspace_size(M, N, code)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.float32, device=x.device)
    qk_rmsnorm_bwd(x, w, rstd, dy, dx, dw, ws, ws_bytes, M, N, code, stream)
    return dx, dw


def xent_bwd(logits, targets, lse, dloss=None, ignore_index=None, z_loss: float = 0.0, stream=None):
    """Cross-entropy backward: dloss * ((1 + 2 z lse) softmax(logits) - onehot(targets))."""
    import torch
    M, N = _rows(logits)
    dx = torch.empty_like(logits)
    qk_xent_bwd_ex(logits, targets, lse, dloss, dx, M, N, _dtype_code(logits), ignore_index, z_loss,
                   stream)
    return dx
