"""Python binding of libnf.so, the GB300 (sm_103a) inner-persistent row
normalization library.

Two layers, both thin:

* ``nf_*`` functions with the C ABI's names and arguments (device pointers
  as ints, a stream handle as an int).  They return the C status code.
* Tensor helpers (``fused_add_rmsnorm``, ``rmsnorm_fwd``, ``layernorm_fwd``,
  ``layernorm_bwd``) that check dtypes/devices/contiguity, take pointers and
  the current CUDA stream from PyTorch, call the C function and raise
  ``NFError`` on a non-OK status.  PyTorch only provides device memory and
  streams; every step of the computation runs in the library's kernels.

There is no fallback: if libnf.so is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnf.so")

NF_OK = 0
NF_ERR_INVALID_ARG = 1
NF_ERR_UNSUPPORTED_HIDDEN = 2
NF_ERR_MISALIGNED = 3
NF_ERR_WORKSPACE_TOO_SMALL = 4
NF_ERR_CUDA = 5
NF_ERR_TIMEOUT = 6
NF_ERR_UNSUPPORTED_PATH = 7

NF_PATH_AUTO, NF_PATH_REG, NF_PATH_CLUSTER, NF_PATH_BULK, NF_PATH_DYNAMIC, NF_PATH_SPLIT, \
    NF_PATH_GRID = 0, 1, 2, 3, 4, 5, 6
PATHS = {"auto": NF_PATH_AUTO, "reg": NF_PATH_REG, "cluster": NF_PATH_CLUSTER, "bulk": NF_PATH_BULK,
         "dynamic": NF_PATH_DYNAMIC, "split": NF_PATH_SPLIT, "grid": NF_PATH_GRID}
PATH_NAMES = {v: k for k, v in PATHS.items()}

NF_OP_FUSED_ADD_RMSNORM, NF_OP_RMSNORM_FWD, NF_OP_LAYERNORM_FWD, NF_OP_LAYERNORM_BWD, \
    NF_OP_RMSNORM_BWD = 0, 1, 2, 3, 4
OPS = {"fused_add_rmsnorm": 0, "rmsnorm_fwd": 1, "layernorm_fwd": 2, "layernorm_bwd": 3,
       "rmsnorm_bwd": 4}

HIDDEN_SET = (1024, 2048, 4096, 5120, 8192, 12288)   # compiled sizes
DYN_MAX_HIDDEN_FWD = 32768    # runtime-hidden path: any multiple of 8 up to these
DYN_MAX_HIDDEN_BWD = 16384
LONG_MAX_HIDDEN_FWD = 262144  # grid-parallel cluster path for longer rows
LONG_MAX_HIDDEN_BWD = 131072
SPLIT_MAX_HIDDEN = 1 << 26    # NF_SPLIT_MAX_HIDDEN: rows across any number of CTAs
GRID_MAX_ROWS = 8             # the grid family (rows held on chip) takes 1 to 8 rows

# Every symbol include/nf.h declares.
EXPORTS = (
    "nf_fused_add_rmsnorm", "nf_rmsnorm_fwd", "nf_layernorm_fwd",
    "nf_layernorm_bwd_workspace_size", "nf_layernorm_bwd",
    "nf_rmsnorm_bwd_workspace_size", "nf_rmsnorm_bwd", "nf_layernorm_bwd_noalloc",
    "nf_outer_norm_workspace_size", "nf_outer_norm_fwd", "nf_outer_norm_bwd",
    "nf_fused_add_rmsnorm_bwd", "nf_workspace_size", "nf_fused_add_rmsnorm_ws", "nf_rmsnorm_fwd_ws",
    "nf_layernorm_fwd_ws",
    "nf_set_path", "nf_plan_query", "nf_plan_compute", "nf_get_device_status",
    "nf_selftest_wait_timeout", "nf_selftest_grid_timeout", "nf_selftest_floor", "nf_status_string",
    "nf_version",
)


class NFError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("grid", ctypes.c_int32), ("block", ctypes.c_int32),
                ("cluster", ctypes.c_int32), ("rows_per_cta", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("partials", ctypes.c_int32)]

    def as_dict(self):
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["path"] = PATH_NAMES.get(d["path"], d["path"])
        return d


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_S = ctypes.c_int


def _bind(lib):
    sig = {
        "nf_fused_add_rmsnorm": (_S, [_P, _P, _P, _I64, _I64, _F, _P]),
        "nf_rmsnorm_fwd": (_S, [_P, _P, _P, _I64, _I64, _F, _P]),
        "nf_layernorm_fwd": (_S, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P]),
        "nf_workspace_size": (ctypes.c_size_t, [ctypes.c_int, _I64, _I64]),
        "nf_fused_add_rmsnorm_ws": (_S, [_P, _P, _P, _I64, _I64, _F, _P, ctypes.c_size_t, _P]),
        "nf_rmsnorm_fwd_ws": (_S, [_P, _P, _P, _I64, _I64, _F, _P, ctypes.c_size_t, _P]),
        "nf_layernorm_fwd_ws": (_S, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P, ctypes.c_size_t, _P]),
        "nf_layernorm_bwd_workspace_size": (ctypes.c_size_t, [_I64, _I64]),
        "nf_layernorm_bwd": (_S, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, ctypes.c_size_t, _P]),
        "nf_rmsnorm_bwd_workspace_size": (ctypes.c_size_t, [_I64, _I64]),
        "nf_rmsnorm_bwd": (_S, [_P, _P, _P, _P, _P, _I64, _I64, _F, _P, ctypes.c_size_t, _P]),
        "nf_layernorm_bwd_noalloc": (_S, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
        "nf_outer_norm_workspace_size": (ctypes.c_size_t, [_I64, _I64]),
        "nf_fused_add_rmsnorm_bwd": (_S, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P, ctypes.c_size_t, _P]),
        "nf_outer_norm_fwd": (_S, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P, ctypes.c_size_t, _P]),
        "nf_outer_norm_bwd": (_S, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, ctypes.c_size_t, _P]),
        "nf_set_path": (_S, [_S]),
        "nf_plan_query": (_S, [_S, _I64, _I64, ctypes.POINTER(Plan)]),
        "nf_plan_compute": (_S, [_S, _I64, _I64, ctypes.c_int32, _S, ctypes.POINTER(Plan)]),
        "nf_get_device_status": (_S, [_P]),
        "nf_selftest_wait_timeout": (_S, [_I64, _P]),
        "nf_selftest_grid_timeout": (_S, [_P, _I64, _P]),
        "nf_selftest_floor": (_S, [ctypes.c_int32, _P, _P, _I64, _P]),
        "nf_status_string": (ctypes.c_char_p, [_S]),
        "nf_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


def lib():
    """The loaded libnf.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m row_normalization_inner_gb300.build` (no fallback exists)")
            _lib = _bind(ctypes.CDLL(LIB_PATH))
        return _lib


def status_string(status: int) -> str:
    return lib().nf_status_string(status).decode()


def version() -> str:
    return lib().nf_version().decode()


# ---------------------------------------------------------------- C-ABI names

def nf_fused_add_rmsnorm(x, residual, weight, rows, hidden, eps, stream) -> int:
    return lib().nf_fused_add_rmsnorm(x, residual, weight, rows, hidden, eps, stream)


def nf_rmsnorm_fwd(y, x, weight, rows, hidden, eps, stream) -> int:
    return lib().nf_rmsnorm_fwd(y, x, weight, rows, hidden, eps, stream)


def nf_workspace_size(op, rows, hidden) -> int:
    return lib().nf_workspace_size(op, rows, hidden)


def nf_fused_add_rmsnorm_ws(x, residual, weight, rows, hidden, eps, workspace, workspace_bytes,
                            stream) -> int:
    return lib().nf_fused_add_rmsnorm_ws(x, residual, weight, rows, hidden, eps, workspace,
                                         workspace_bytes, stream)


def nf_rmsnorm_fwd_ws(y, x, weight, rows, hidden, eps, workspace, workspace_bytes, stream) -> int:
    return lib().nf_rmsnorm_fwd_ws(y, x, weight, rows, hidden, eps, workspace, workspace_bytes,
                                   stream)


def nf_layernorm_fwd_ws(y, mean, rstd, x, gamma, beta, rows, hidden, eps, workspace,
                        workspace_bytes, stream) -> int:
    return lib().nf_layernorm_fwd_ws(y, mean, rstd, x, gamma, beta, rows, hidden, eps, workspace,
                                     workspace_bytes, stream)


def nf_layernorm_fwd(y, mean, rstd, x, gamma, beta, rows, hidden, eps, stream) -> int:
    return lib().nf_layernorm_fwd(y, mean, rstd, x, gamma, beta, rows, hidden, eps, stream)


def nf_layernorm_bwd_workspace_size(rows, hidden) -> int:
    return lib().nf_layernorm_bwd_workspace_size(rows, hidden)


def nf_layernorm_bwd(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden, workspace,
                     workspace_bytes, stream) -> int:
    return lib().nf_layernorm_bwd(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden,
                                  workspace, workspace_bytes, stream)


def nf_rmsnorm_bwd_workspace_size(rows, hidden) -> int:
    return lib().nf_rmsnorm_bwd_workspace_size(rows, hidden)


def nf_rmsnorm_bwd(dx, dw, dy, x, weight, rows, hidden, eps, workspace, workspace_bytes,
                   stream) -> int:
    return lib().nf_rmsnorm_bwd(dx, dw, dy, x, weight, rows, hidden, eps, workspace,
                                workspace_bytes, stream)


def nf_layernorm_bwd_noalloc(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden,
                             stream) -> int:
    return lib().nf_layernorm_bwd_noalloc(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows,
                                          hidden, stream)


NOALLOC_SCRATCH_BYTES = 16 << 20  # NF_LAYERNORM_BWD_NOALLOC_SCRATCH_BYTES


def nf_fused_add_rmsnorm_bwd(dx, dw, dy, dres, residual, weight, rows, hidden, eps, workspace,
                             workspace_bytes, stream) -> int:
    return lib().nf_fused_add_rmsnorm_bwd(dx, dw, dy, dres, residual, weight, rows, hidden, eps,
                                          workspace, workspace_bytes, stream)


def nf_outer_norm_workspace_size(rows, hidden) -> int:
    return lib().nf_outer_norm_workspace_size(rows, hidden)


def nf_outer_norm_fwd(y, mean, rstd, x, gamma, beta, rows, hidden, eps, workspace,
                      workspace_bytes, stream) -> int:
    return lib().nf_outer_norm_fwd(y, mean, rstd, x, gamma, beta, rows, hidden, eps, workspace,
                                   workspace_bytes, stream)


def nf_outer_norm_bwd(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden, workspace,
                      workspace_bytes, stream) -> int:
    return lib().nf_outer_norm_bwd(dx, dgamma, dbeta, dy, x, mean, rstd, gamma, rows, hidden,
                                   workspace, workspace_bytes, stream)


def nf_set_path(path) -> int:
    if isinstance(path, str):
        path = PATHS[path]
    return lib().nf_set_path(path)


def nf_plan_query(op, rows, hidden) -> dict:
    if isinstance(op, str):
        op = OPS[op]
    p = Plan()
    st = lib().nf_plan_query(op, rows, hidden, ctypes.byref(p))
    if st != NF_OK:
        raise NFError(st, "nf_plan_query")
    return p.as_dict()


def nf_plan_compute(op, rows, hidden, sm_count, path=NF_PATH_AUTO):
    """Pure host planning.  Returns (status, plan dict or None)."""
    if isinstance(op, str):
        op = OPS[op]
    if isinstance(path, str):
        path = PATHS[path]
    p = Plan()
    st = lib().nf_plan_compute(op, rows, hidden, sm_count, path, ctypes.byref(p))
    return st, (p.as_dict() if st == NF_OK else None)


def nf_get_device_status(stream) -> int:
    return lib().nf_get_device_status(stream)


def nf_selftest_wait_timeout(timeout_ns, stream) -> int:
    return lib().nf_selftest_wait_timeout(timeout_ns, stream)


def nf_selftest_grid_timeout(workspace, timeout_ns, stream) -> int:
    return lib().nf_selftest_grid_timeout(workspace, timeout_ns, stream)


def nf_selftest_floor(kind, dst, src, nbytes, stream) -> int:
    return lib().nf_selftest_floor(kind, dst, src, nbytes, stream)


# ---------------------------------------------------------------- tensor helpers

def _check(st: int, where: str):
    if st != NF_OK:
        raise NFError(st, where)


def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _rows_hidden(x):
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    return rows, hidden


def _fwd_workspace(op, rows, hidden, device, workspace):
    """(pointer, bytes) of the workspace a forward call needs now: a caller
    tensor if given, else one allocated here (by PyTorch) only when the
    plan is the split or grid family."""
    import torch
    if workspace is not None:
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if rows == 0 or nf_plan_query(op, rows, hidden)["path"] not in ("split", "grid"):
        return None, 0
    n = nf_workspace_size(OPS[op], rows, hidden)
    # freed right after the launch: PyTorch's allocator hands the block to
    # later work on the same stream only, which runs after these kernels
    t = torch.empty(max(n, 16), dtype=torch.uint8, device=device)
    return t.data_ptr(), n


def fused_add_rmsnorm(x, residual, weight, eps: float = 1e-6, stream=None, workspace=None):
    """In place: residual += x; x = rmsnorm(residual) * weight.  Returns (x, residual)."""
    import torch
    for t, n in ((x, "x"), (residual, "residual"), (weight, "weight")):
        _need(t, torch.bfloat16, n)
    rows, hidden = _rows_hidden(x)
    if residual.shape != x.shape or weight.shape != (hidden,):
        raise ValueError("shape mismatch")
    wp, wb = _fwd_workspace("fused_add_rmsnorm", rows, hidden, x.device, workspace)
    _check(nf_fused_add_rmsnorm_ws(x.data_ptr(), residual.data_ptr(), weight.data_ptr(), rows,
                                   hidden, eps, wp, wb, _stream(stream)), "nf_fused_add_rmsnorm_ws")
    return x, residual


def rmsnorm_fwd(x, weight, eps: float = 1e-6, out=None, stream=None, workspace=None):
    import torch
    _need(x, torch.bfloat16, "x")
    _need(weight, torch.bfloat16, "weight")
    rows, hidden = _rows_hidden(x)
    y = torch.empty_like(x) if out is None else out
    _need(y, torch.bfloat16, "out")
    wp, wb = _fwd_workspace("rmsnorm_fwd", rows, hidden, x.device, workspace)
    _check(nf_rmsnorm_fwd_ws(y.data_ptr(), x.data_ptr(), weight.data_ptr(), rows, hidden, eps,
                             wp, wb, _stream(stream)), "nf_rmsnorm_fwd_ws")
    return y


def layernorm_fwd(x, gamma, beta, eps: float = 1e-5, out=None, stream=None, workspace=None):
    """Returns (y bf16, mean fp32 [rows], rstd fp32 [rows])."""
    import torch
    for t, n in ((x, "x"), (gamma, "gamma"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    rows, hidden = _rows_hidden(x)
    y = torch.empty_like(x) if out is None else out
    mean = torch.empty(rows, dtype=torch.float32, device=x.device)
    rstd = torch.empty(rows, dtype=torch.float32, device=x.device)
    wp, wb = _fwd_workspace("layernorm_fwd", rows, hidden, x.device, workspace)
    _check(nf_layernorm_fwd_ws(y.data_ptr(), mean.data_ptr(), rstd.data_ptr(), x.data_ptr(),
                               gamma.data_ptr(), beta.data_ptr(), rows, hidden, eps, wp, wb,
                               _stream(stream)), "nf_layernorm_fwd_ws")
    return y, mean, rstd


def layernorm_bwd(dy, x, mean, rstd, gamma, workspace=None, out=None, stream=None):
    """Returns (dx bf16, dgamma fp32, dbeta fp32).  The workspace is
    allocated here (by PyTorch) when not given; the library never allocates."""
    import torch
    for t, n in ((dy, "dy"), (x, "x"), (gamma, "gamma")):
        _need(t, torch.bfloat16, n)
    _need(mean, torch.float32, "mean")
    _need(rstd, torch.float32, "rstd")
    rows, hidden = _rows_hidden(x)
    dx = torch.empty_like(x) if out is None else out
    dgamma = torch.empty(hidden, dtype=torch.float32, device=x.device)
    dbeta = torch.empty(hidden, dtype=torch.float32, device=x.device)
    need = nf_layernorm_bwd_workspace_size(rows, hidden)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(nf_layernorm_bwd(dx.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(), dy.data_ptr(),
                            x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), gamma.data_ptr(), rows,
                            hidden, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            _stream(stream)), "nf_layernorm_bwd")
    return dx, dgamma, dbeta


def rmsnorm_bwd(dy, x, weight, eps: float = 1e-6, workspace=None, out=None, stream=None):
    """Returns (dx bf16, dw fp32).  rstd is recomputed from x in the kernel."""
    import torch
    for t, n in ((dy, "dy"), (x, "x"), (weight, "weight")):
        _need(t, torch.bfloat16, n)
    rows, hidden = _rows_hidden(x)
    dx = torch.empty_like(x) if out is None else out
    dw = torch.empty(hidden, dtype=torch.float32, device=x.device)
    need = nf_rmsnorm_bwd_workspace_size(rows, hidden)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(nf_rmsnorm_bwd(dx.data_ptr(), dw.data_ptr(), dy.data_ptr(), x.data_ptr(),
                          weight.data_ptr(), rows, hidden, eps, workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(), _stream(stream)),
           "nf_rmsnorm_bwd")
    return dx, dw


def fused_add_rmsnorm_bwd(dy, residual, weight, dres=None, eps: float = 1e-6, workspace=None,
                         out=None, stream=None):
    """Backward of fused_add_rmsnorm given the saved residual output.
    Returns (dx bf16 -- the gradient of both x and residual --, dw fp32)."""
    import torch
    for t, n in ((dy, "dy"), (residual, "residual"), (weight, "weight")):
        _need(t, torch.bfloat16, n)
    if dres is not None:
        _need(dres, torch.bfloat16, "dres")
    rows, hidden = _rows_hidden(residual)
    dx = torch.empty_like(residual) if out is None else out
    dw = torch.empty(hidden, dtype=torch.float32, device=residual.device)
    need = nf_rmsnorm_bwd_workspace_size(rows, hidden)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=residual.device)
    _check(nf_fused_add_rmsnorm_bwd(dx.data_ptr(), dw.data_ptr(), dy.data_ptr(),
                                    None if dres is None else dres.data_ptr(),
                                    residual.data_ptr(), weight.data_ptr(), rows, hidden, eps,
                                    workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "nf_fused_add_rmsnorm_bwd")
    return dx, dw


def outer_norm_fwd(x, gamma, beta, eps: float = 1e-5, workspace=None, out=None, stream=None):
    """Per-column normalization over the rows.  Returns (y, mean [hidden], rstd [hidden])."""
    import torch
    for t, n in ((x, "x"), (gamma, "gamma"), (beta, "beta")):
        _need(t, torch.bfloat16, n)
    rows, hidden = _rows_hidden(x)
    y = torch.empty_like(x) if out is None else out
    mean = torch.empty(hidden, dtype=torch.float32, device=x.device)
    rstd = torch.empty(hidden, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(nf_outer_norm_workspace_size(rows, hidden), 16),
                                dtype=torch.uint8, device=x.device)
    _check(nf_outer_norm_fwd(y.data_ptr(), mean.data_ptr(), rstd.data_ptr(), x.data_ptr(),
                             gamma.data_ptr(), beta.data_ptr(), rows, hidden, eps,
                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                             _stream(stream)), "nf_outer_norm_fwd")
    return y, mean, rstd


def outer_norm_bwd(dy, x, mean, rstd, gamma, workspace=None, out=None, stream=None):
    """Returns (dx bf16, dgamma fp32, dbeta fp32)."""
    import torch
    for t, n in ((dy, "dy"), (x, "x"), (gamma, "gamma")):
        _need(t, torch.bfloat16, n)
    _need(mean, torch.float32, "mean")
    _need(rstd, torch.float32, "rstd")
    rows, hidden = _rows_hidden(x)
    dx = torch.empty_like(x) if out is None else out
    dgamma = torch.empty(hidden, dtype=torch.float32, device=x.device)
    dbeta = torch.empty(hidden, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(nf_outer_norm_workspace_size(rows, hidden), 16),
                                dtype=torch.uint8, device=x.device)
    _check(nf_outer_norm_bwd(dx.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(), dy.data_ptr(),
                             x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), gamma.data_ptr(),
                             rows, hidden, workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream(stream)),
           "nf_outer_norm_bwd")
    return dx, dgamma, dbeta


def set_path(path):
    _check(nf_set_path(path), "nf_set_path")


class forced_path:
    """Context manager: force a kernel family, restore AUTO on exit."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        set_path(self.path)
        return self

    def __exit__(self, *exc):
        set_path(NF_PATH_AUTO)
