"""fp64 CPU oracle for the row-normalization path (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm import this package.  The product library never
does, and this package imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, straight loops); this
module only builds it with gcc, loads it with ctypes and marshals arrays.
Inputs are bf16 tensors (torch, CPU) or numpy uint16 arrays of bf16 bit
patterns; they are widened exactly to float64 before any arithmetic.
Every function returns float64 numpy arrays (unrounded); ``to_bf16`` rounds
a float64 array to bf16 bit patterns (one rounding, ties to even).

Operations and where the pages name them:
  fused_add_rmsnorm  -- "optimize inner persistent scheduler for static
                        fusion" (NVIDIA/Fuser PR #5281), changes walkthrough,
                        FlashInfer RMSNormAdd benchmark with in-place update.
  rmsnorm_fwd,
  layernorm_fwd      -- "TMA inner persistent scheduler" (NVIDIA/Fuser
                        PR #5587), description: RMS norm and layer norm.
  layernorm_bwd      -- "Llu/ln bwd" (NVIDIA/Fuser PR #207): layer norm
                        backward, a combined inner + outer reduction.
  rmsnorm_bwd        -- the RMS norm counterpart of the same combined
                        reduction ("TMA inner persistent scheduler",
                        description: RMS norm, with a workspace).
  outer_norm_fwd,
  outer_norm_bwd     -- outer normalization (statistics per column, over the
                        rows), listed among the normalization variants in
                        the "Llu/ln bwd" discussion.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_U16 = ctypes.POINTER(ctypes.c_uint16)
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, ISO C, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    lib.or_bf16_to_double_array.argtypes = [_U16, _D, _I64]
    lib.or_double_to_bf16_array.argtypes = [_D, _U16, _I64]
    lib.or_rmsnorm_fwd.argtypes = [_D, _D, _I64, _I64, ctypes.c_double, _D, _D]
    lib.or_fused_add_rmsnorm.argtypes = [_D, _D, _D, _I64, _I64, ctypes.c_double,
                                         ctypes.c_int, _D, _D, _D]
    lib.or_layernorm_fwd.argtypes = [_D, _D, _D, _I64, _I64, ctypes.c_double, _D, _D, _D]
    lib.or_layernorm_bwd.argtypes = [_D, _D, _D, _D, _D, _I64, _I64, _D, _D, _D]
    lib.or_rmsnorm_bwd.argtypes = [_D, _D, _D, _D, _I64, _I64, _D, _D]
    lib.or_fused_add_rmsnorm_bwd.argtypes = [_D, _D, _D, _D, _I64, _I64, ctypes.c_double, _D, _D]
    lib.or_outer_norm_fwd.argtypes = [_D, _D, _D, _I64, _I64, ctypes.c_double, _D, _D, _D]
    lib.or_outer_norm_bwd.argtypes = [_D, _D, _D, _D, _D, _I64, _I64, _D, _D, _D]
    for f in (lib.or_bf16_to_double_array, lib.or_double_to_bf16_array, lib.or_rmsnorm_fwd,
              lib.or_fused_add_rmsnorm, lib.or_layernorm_fwd, lib.or_layernorm_bwd,
              lib.or_rmsnorm_bwd, lib.or_fused_add_rmsnorm_bwd, lib.or_outer_norm_fwd,
              lib.or_outer_norm_bwd):
        f.restype = None
    return lib


def _load():
    """Load liboracle.so.  ORACLE_LIBRARY names another build of oracle.c
    instead; the mutation tests use it to load copies with a planted mistake
    and check that some pin fails."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ORACLE_LIBRARY") or build()
            _lib = _bind(ctypes.CDLL(path))
        return _lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _bits(t) -> np.ndarray:
    """bf16 bit patterns as a contiguous numpy uint16 array (keeps the shape)."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16, t.dtype
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def widen(t) -> np.ndarray:
    """bf16 (torch tensor or uint16 bit array) -> float64, exactly."""
    b = _bits(t)
    out = np.empty(b.shape, dtype=np.float64)
    _load().or_bf16_to_double_array(b.ctypes.data_as(_U16), _dp(out), b.size)
    return out


def to_bf16(a: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().or_double_to_bf16_array(_dp(a), out.ctypes.data_as(_U16), a.size)
    return out


def bf16_value(a: np.ndarray) -> np.ndarray:
    """float64 -> the float64 value of its bf16 rounding."""
    return widen(to_bf16(a))


def _f64(a, shape=None) -> np.ndarray:
    """A float64 contiguous copy; bf16 inputs are widened exactly."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.dtype == torch.bfloat16:
                a = widen(a)
            else:
                a = a.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    if isinstance(a, np.ndarray) and a.dtype == np.uint16:
        a = widen(a)
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None:
        a = a.reshape(shape)
    return a


def rmsnorm_fwd(x, w, eps: float):
    """y = x / sqrt(mean(x^2) + eps) * w per row.  Returns (y, rstd)."""
    x = _f64(x)
    rows, hidden = x.shape
    w = _f64(w, (hidden,))
    y = np.empty_like(x)
    rstd = np.empty(rows, dtype=np.float64)
    _load().or_rmsnorm_fwd(_dp(x), _dp(w), rows, hidden, float(eps), _dp(y), _dp(rstd))
    return y, rstd


def fused_add_rmsnorm(x, residual, w, eps: float, normalize_rounded: bool = False):
    """residual <- residual + x ; x <- rmsnorm(residual) * w.

    Returns (residual_out, x_out, rstd) in float64, unrounded.  With
    ``normalize_rounded`` the normalization reads bf16(residual + x)."""
    x = _f64(x)
    rows, hidden = x.shape
    r = _f64(residual, (rows, hidden))
    w = _f64(w, (hidden,))
    s = np.empty_like(x)
    y = np.empty_like(x)
    rstd = np.empty(rows, dtype=np.float64)
    _load().or_fused_add_rmsnorm(_dp(x), _dp(r), _dp(w), rows, hidden, float(eps),
                                 1 if normalize_rounded else 0, _dp(s), _dp(y), _dp(rstd))
    return s, y, rstd


def layernorm_fwd(x, gamma, beta, eps: float):
    """y = (x - mean) * rstd * gamma + beta (biased variance).  Returns (y, mean, rstd)."""
    x = _f64(x)
    rows, hidden = x.shape
    g = _f64(gamma, (hidden,))
    b = _f64(beta, (hidden,))
    y = np.empty_like(x)
    mean = np.empty(rows, dtype=np.float64)
    rstd = np.empty(rows, dtype=np.float64)
    _load().or_layernorm_fwd(_dp(x), _dp(g), _dp(b), rows, hidden, float(eps),
                             _dp(y), _dp(mean), _dp(rstd))
    return y, mean, rstd


def layernorm_bwd(dy, x, mean, rstd, gamma):
    """Gradients of sum(dy * LayerNorm(x)) given the saved mean/rstd.

    Returns (dx, dgamma, dbeta) in float64."""
    x = _f64(x)
    rows, hidden = x.shape
    dy = _f64(dy, (rows, hidden))
    mean = _f64(mean, (rows,))
    rstd = _f64(rstd, (rows,))
    g = _f64(gamma, (hidden,))
    dx = np.empty_like(x)
    dgamma = np.empty(hidden, dtype=np.float64)
    dbeta = np.empty(hidden, dtype=np.float64)
    _load().or_layernorm_bwd(_dp(dy), _dp(x), _dp(mean), _dp(rstd), _dp(g), rows, hidden,
                             _dp(dx), _dp(dgamma), _dp(dbeta))
    return dx, dgamma, dbeta


def rmsnorm_bwd(dy, x, rstd, w):
    """Gradients of sum(dy * RMSNorm(x) * w) given the saved rstd.

    Returns (dx, dw) in float64."""
    x = _f64(x)
    rows, hidden = x.shape
    dy = _f64(dy, (rows, hidden))
    rstd = _f64(rstd, (rows,))
    w = _f64(w, (hidden,))
    dx = np.empty_like(x)
    dw = np.empty(hidden, dtype=np.float64)
    _load().or_rmsnorm_bwd(_dp(dy), _dp(x), _dp(rstd), _dp(w), rows, hidden, _dp(dx), _dp(dw))
    return dx, dw


def fused_add_rmsnorm_bwd(dy, dres, s, w, eps: float):
    """Backward of the fused residual add + RMSNorm, given the saved residual
    output s and the gradients dy (normalized output) and dres (residual
    stream, or None).  Returns (ds, dw) in float64: ds is the gradient of
    both x and residual."""
    s = _f64(s)
    rows, hidden = s.shape
    dy = _f64(dy, (rows, hidden))
    w = _f64(w, (hidden,))
    ds = np.empty_like(s)
    dw = np.empty(hidden, dtype=np.float64)
    pr = None
    if dres is not None:
        dres = _f64(dres, (rows, hidden))
        pr = _dp(dres)
    _load().or_fused_add_rmsnorm_bwd(_dp(dy), pr, _dp(s), _dp(w), rows, hidden, float(eps),
                                     _dp(ds), _dp(dw))
    return ds, dw


def outer_norm_fwd(x, gamma, beta, eps: float):
    """Per-column normalization over the rows (biased variance).

    Returns (y [rows, hidden], mean [hidden], rstd [hidden]) in float64."""
    x = _f64(x)
    rows, hidden = x.shape
    g = _f64(gamma, (hidden,))
    b = _f64(beta, (hidden,))
    y = np.empty_like(x)
    mean = np.empty(hidden, dtype=np.float64)
    rstd = np.empty(hidden, dtype=np.float64)
    _load().or_outer_norm_fwd(_dp(x), _dp(g), _dp(b), rows, hidden, float(eps),
                              _dp(y), _dp(mean), _dp(rstd))
    return y, mean, rstd


def outer_norm_bwd(dy, x, mean, rstd, gamma):
    """Gradients of sum(dy * OuterNorm(x)) given the saved per-column mean/rstd.

    Returns (dx, dgamma, dbeta) in float64."""
    x = _f64(x)
    rows, hidden = x.shape
    dy = _f64(dy, (rows, hidden))
    mean = _f64(mean, (hidden,))
    rstd = _f64(rstd, (hidden,))
    g = _f64(gamma, (hidden,))
    dx = np.empty_like(x)
    dgamma = np.empty(hidden, dtype=np.float64)
    dbeta = np.empty(hidden, dtype=np.float64)
    _load().or_outer_norm_bwd(_dp(dy), _dp(x), _dp(mean), _dp(rstd), _dp(g), rows, hidden,
                              _dp(dx), _dp(dgamma), _dp(dbeta))
    return dx, dgamma, dbeta
