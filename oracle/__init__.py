"""fp64 CPU oracle for softmax / RMSNorm / cross-entropy forward.

TEST INFRASTRUCTURE ONLY.  The arithmetic lives in ``oracle.c`` (plain C,
double precision, one row at a time); this module compiles it with gcc and
marshals numpy arrays through ctypes.  Only the test suite, the smoke check and
the benchmark's CPU-baseline leg may import this package.  The CUDA library
never imports, links or calls it, and this package imports nothing from the
CUDA library.

Every function takes and returns float64 numpy arrays.  Inputs in fp32 or bf16
must be widened to float64 by the caller (an exact conversion); nothing here
rounds to a narrower type.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(_BUILD_DIR, "liboracle.so")

# No fused multiply-add contraction, no fast-math: the same doubles on any host.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def compile_library(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile ``source`` into the shared library ``output`` with gcc."""
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = output + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, source, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, output)
    return output


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` unless an up-to-date library is already present."""
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_library()
    return LIBRARY


def bind(path: str):
    """Load a compiled oracle library and declare its three entry points."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_softmax_fwd.argtypes = [dp, dp, i64, i64]
    lib.oracle_softmax_fwd.restype = None
    lib.oracle_rmsnorm_fwd.argtypes = [dp, dp, dp, dp, i64, i64, ctypes.c_double]
    lib.oracle_rmsnorm_fwd.restype = None
    lib.oracle_xent_fwd.argtypes = [dp, lp, dp, dp, i64, i64]
    lib.oracle_xent_fwd.restype = None
    lib.oracle_softmax_bwd.argtypes = [dp, dp, dp, i64, i64]
    lib.oracle_softmax_bwd.restype = None
    lib.oracle_rmsnorm_bwd.argtypes = [dp, dp, dp, dp, dp, dp, i64, i64]
    lib.oracle_rmsnorm_bwd.restype = None
    lib.oracle_xent_bwd.argtypes = [dp, lp, dp, dp, dp, i64, i64]
    lib.oracle_xent_bwd.restype = None
    lib.oracle_xent_fwd_ex.argtypes = [dp, lp, dp, dp, dp, i64, i64, ctypes.c_int, i64, ctypes.c_double]
    lib.oracle_xent_fwd_ex.restype = None
    lib.oracle_xent_bwd_ex.argtypes = [dp, lp, dp, dp, dp, i64, i64, ctypes.c_int, i64, ctypes.c_double]
    lib.oracle_xent_bwd_ex.restype = None
    lib.oracle_layernorm_fwd.argtypes = [dp, dp, dp, dp, dp, dp, i64, i64, ctypes.c_double]
    lib.oracle_layernorm_fwd.restype = None
    return lib


def library():
    """The process-wide oracle library, compiled on first use."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
        return _lib


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a


def _ptr(a: np.ndarray, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def softmax_fwd(x, lib=None) -> np.ndarray:
    """Row-wise softmax of a 2-D float64 array (M x N)."""
    lib = lib or library()
    x = _f64(x)
    M, N = x.shape
    y = np.empty_like(x)
    lib.oracle_softmax_fwd(_ptr(x), _ptr(y), M, N)
    return y


def rmsnorm_fwd(x, w, eps: float, lib=None):
    """Row-wise RMSNorm of a 2-D float64 array; returns (y, rstd)."""
    lib = lib or library()
    x = _f64(x)
    w = _f64(w)
    M, N = x.shape
    if w.shape != (N,):
        raise ValueError(f"w must have shape ({N},), got {w.shape}")
    y = np.empty_like(x)
    rstd = np.empty(M, dtype=np.float64)
    lib.oracle_rmsnorm_fwd(_ptr(x), _ptr(w), _ptr(y), _ptr(rstd), M, N, float(eps))
    return y, rstd


def xent_fwd(x, target, lib=None):
    """Row-wise cross-entropy of logits x (M x N) against int64 targets [M];
    returns (loss, lse)."""
    lib = lib or library()
    x = _f64(x)
    M, N = x.shape
    t = np.ascontiguousarray(target, dtype=np.int64)
    if t.shape != (M,):
        raise ValueError(f"target must have shape ({M},), got {t.shape}")
    loss = np.empty(M, dtype=np.float64)
    lse = np.empty(M, dtype=np.float64)
    lib.oracle_xent_fwd(_ptr(x), _ptr(t, ctypes.c_int64), _ptr(loss), _ptr(lse), M, N)
    return loss, lse


def softmax_bwd(y, dy, lib=None) -> np.ndarray:
    """dx of softmax given its output y and the upstream gradient dy (M x N)."""
    lib = lib or library()
    y, dy = _f64(y), _f64(dy)
    M, N = y.shape
    if dy.shape != (M, N):
        raise ValueError("y and dy must have the same shape")
    dx = np.empty_like(y)
    lib.oracle_softmax_bwd(_ptr(y), _ptr(dy), _ptr(dx), M, N)
    return dx


def rmsnorm_bwd(x, w, rstd, dy, lib=None):
    """(dx, dw) of RMSNorm given x, w, the forward rstd and the upstream dy."""
    lib = lib or library()
    x, w, rstd, dy = _f64(x), _f64(w), _f64(rstd), _f64(dy)
    M, N = x.shape
    if w.shape != (N,) or rstd.shape != (M,) or dy.shape != (M, N):
        raise ValueError("shapes: x [M, N], w [N], rstd [M], dy [M, N]")
    dx = np.empty_like(x)
    dw = np.empty(N, dtype=np.float64)
    lib.oracle_rmsnorm_bwd(_ptr(x), _ptr(w), _ptr(rstd), _ptr(dy), _ptr(dx), _ptr(dw), M, N)
    return dx, dw


def xent_bwd(x, target, lse, dloss, lib=None) -> np.ndarray:
    """dlogits of the per-row cross-entropy given the forward lse and dloss [M]."""
    lib = lib or library()
    x, lse, dloss = _f64(x), _f64(lse), _f64(dloss)
    M, N = x.shape
    t = np.ascontiguousarray(target, dtype=np.int64)
    if t.shape != (M,) or lse.shape != (M,) or dloss.shape != (M,):
        raise ValueError("shapes: x [M, N], target/lse/dloss [M]")
    dx = np.empty_like(x)
    lib.oracle_xent_bwd(_ptr(x), _ptr(t, ctypes.c_int64), _ptr(lse), _ptr(dloss), _ptr(dx), M, N)
    return dx


def _ignore_args(ignore_index):
    """(has_ignore, ignore_index) for the C oracle: None means no row is
    ignored.  The index passed with the flag off is INT64_MIN, the value a
    sentinel would use, so an oracle that tested the index alone would be
    caught by the extreme-target pins."""
    return (0, -(2 ** 63)) if ignore_index is None else (1, int(ignore_index))


def xent_fwd_ex(x, target, ignore_index=None, z: float = 0.0, lib=None):
    """Cross-entropy with an ignore index (None: no row is ignored) and a
    z-loss term; returns (loss [M], lse [M], mean over the rows not ignored)."""
    lib = lib or library()
    x = _f64(x)
    M, N = x.shape
    t = np.ascontiguousarray(target, dtype=np.int64)
    loss = np.empty(M, dtype=np.float64)
    lse = np.empty(M, dtype=np.float64)
    mean = np.empty(1, dtype=np.float64)
    lib.oracle_xent_fwd_ex(_ptr(x), _ptr(t, ctypes.c_int64), _ptr(loss), _ptr(lse), _ptr(mean), M, N,
                           *_ignore_args(ignore_index), float(z))
    return loss, lse, float(mean[0])


def xent_bwd_ex(x, target, lse, dloss, ignore_index=None, z: float = 0.0, lib=None):
    """dlogits of xent_fwd_ex's per-row loss, given the forward lse and dloss [M]."""
    lib = lib or library()
    x, lse, dloss = _f64(x), _f64(lse), _f64(dloss)
    M, N = x.shape
    t = np.ascontiguousarray(target, dtype=np.int64)
    dx = np.empty_like(x)
    lib.oracle_xent_bwd_ex(_ptr(x), _ptr(t, ctypes.c_int64), _ptr(lse), _ptr(dloss), _ptr(dx), M, N,
                           *_ignore_args(ignore_index), float(z))
    return dx


def layernorm_fwd(x, w, b, eps: float, lib=None):
    """Row-wise LayerNorm (population variance, eps inside the root); b may be
    None.  Returns (y, mean, rstd)."""
    lib = lib or library()
    x, w = _f64(x), _f64(w)
    M, N = x.shape
    bb = None if b is None else _f64(b)
    if w.shape != (N,) or (bb is not None and bb.shape != (N,)):
        raise ValueError("w and b must have shape (N,)")
    y = np.empty_like(x)
    mean = np.empty(M, dtype=np.float64)
    rstd = np.empty(M, dtype=np.float64)
    lib.oracle_layernorm_fwd(_ptr(x), _ptr(w), None if bb is None else _ptr(bb), _ptr(y), _ptr(mean),
                             _ptr(rstd), M, N, float(eps))
    return y, mean, rstd
