"""Python binding of the fused normalization library (``libnormfuse.so``).

The functions here have the names of the C entry points declared in
``include/normfuse.h`` and only marshal arguments: torch tensors become
device pointers, the torch stream becomes a ``cudaStream_t``, and the return
status becomes an exception. Every step of the computation runs in the CUDA
kernels of the library; there is no fallback. If the library has not been
built, loading it raises.

PyTorch is used for device memory and streams only.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH, build as build_library

__all__ = [
    "LN_F32", "LN_BF16", "LN_F16", "LN_LAYERNORM", "LN_RMSNORM", "NormError",
    "LN_OK", "LN_ERR_NULL", "LN_ERR_ALIGN", "LN_ERR_SHAPE", "LN_ERR_UNSUPPORTED",
    "LN_ERR_CUDA", "LN_ERR_WORKSPACE", "LN_ERR_INVALID", "LN_ERR_SCRATCH_LIMIT",
    "LN_NOALLOC_SCRATCH_BYTES",
    "load_library", "build_library", "ln_fwd", "ln_fwd_ex", "ln_bwd", "ln_bwd_ex",
    "ln_bwd_workspace_bytes",
    "ln_status_string", "ln_last_cuda_error", "ln_device_error", "ln_bwd_noalloc",
    "ln_testing_select_kernels", "ln_testing_plan", "exported_symbols", "ln_fwd_from_partials",
    "LN_PARTIALS_SUM_SQ", "LN_PARTIALS_SUM_M2", "fused_norm_fwd_from_partials",
    "fused_norm_fwd", "fused_norm_bwd", "Workspace",
]

# Mirrors of include/normfuse.h (a CPU test checks them against the header).
LN_F32, LN_BF16, LN_F16 = 0, 1, 2
LN_LAYERNORM, LN_RMSNORM = 0, 1
(LN_OK, LN_ERR_NULL, LN_ERR_ALIGN, LN_ERR_SHAPE, LN_ERR_UNSUPPORTED, LN_ERR_CUDA,
 LN_ERR_WORKSPACE, LN_ERR_INVALID, LN_ERR_SCRATCH_LIMIT) = range(9)
LN_NOALLOC_SCRATCH_BYTES = 16 << 20
LN_PARTIALS_SUM_SQ, LN_PARTIALS_SUM_M2 = 0, 1
_PARTIAL_CODES = {"sum_sq": LN_PARTIALS_SUM_SQ, "sum_m2": LN_PARTIALS_SUM_M2,
                  LN_PARTIALS_SUM_SQ: LN_PARTIALS_SUM_SQ, LN_PARTIALS_SUM_M2: LN_PARTIALS_SUM_M2}
_DTYPE_CODES = {torch.float32: LN_F32, torch.bfloat16: LN_BF16, torch.float16: LN_F16}
_MODE_CODES = {"layernorm": LN_LAYERNORM, "rmsnorm": LN_RMSNORM,
               LN_LAYERNORM: LN_LAYERNORM, LN_RMSNORM: LN_RMSNORM}

_lib = None
_lock = threading.Lock()


class NormError(RuntimeError):
    """A non-zero ``ln_status`` returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        msg = ln_status_string(status)
        if status == 5:
            msg += f" (cudaError {ln_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load ``libnormfuse.so`` (built in-tree by ``build_library()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.isfile(path):
            raise RuntimeError(
                f"CUDA library not built: {path} is missing. "
                "Run `python -m normalization_fwd_gb300.build` (needs nvcc).")
        lib = ctypes.CDLL(path)
        vp, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        ci = ctypes.c_int
        lib.ln_fwd.argtypes = [vp, vp, vp, vp, vp, f32, ci, ci, vp, vp, vp, vp, vp, vp,
                               i64, i64, ci]
        lib.ln_fwd.restype = ci
        lib.ln_fwd_ex.argtypes = [vp, vp, vp, vp, vp, f32, ci, ci, vp, vp, vp, vp, vp, vp, vp,
                                  vp, i64, i64, ci]
        lib.ln_fwd_ex.restype = ci
        lib.ln_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, ci, ci,
                               vp, sz]
        lib.ln_bwd.restype = ci
        lib.ln_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, ci, ci,
                                  vp, sz, ci]
        lib.ln_bwd_ex.restype = ci
        lib.ln_bwd_workspace_bytes.argtypes = [i64, i64, ci, ci, ctypes.POINTER(sz)]
        lib.ln_bwd_workspace_bytes.restype = ci
        lib.ln_status_string.argtypes = [ci]
        lib.ln_status_string.restype = ctypes.c_char_p
        lib.ln_last_cuda_error.argtypes = []
        lib.ln_last_cuda_error.restype = ci
        lib.ln_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
        lib.ln_device_error.restype = ci
        lib.ln_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, ci, ci]
        lib.ln_bwd_noalloc.restype = ci
        lib.ln_softmax_fwd.argtypes = [vp, vp, vp, i64, i64, ci]
        lib.ln_softmax_fwd.restype = ci
        lib.ln_fwd_from_partials.argtypes = [vp, vp, vp, i64, i64, ci, vp, vp, f32, ci, ci, vp,
                                             vp, vp, vp, vp, i64, i64, ci]
        lib.ln_fwd_from_partials.restype = ci
        lib.ln_testing_select_kernels.argtypes = [ci, ci, ci]
        lib.ln_testing_select_kernels.restype = ci
        lib.ln_testing_plan.argtypes = [ci, i64, i64, ci, ci, ci, ctypes.POINTER(ci)]
        lib.ln_testing_plan.restype = ci
        _lib = lib
        return lib


def exported_symbols() -> list[str]:
    """Names of the C entry points this binding wraps."""
    return ["ln_fwd", "ln_fwd_ex", "ln_bwd", "ln_bwd_ex", "ln_bwd_workspace_bytes",
            "ln_status_string", "ln_last_cuda_error", "ln_device_error", "ln_bwd_noalloc",
            "ln_softmax_fwd", "ln_testing_select_kernels", "ln_fwd_from_partials",
            "ln_testing_plan"]


_FAMILY_CODES = {"default": 0, "ring": 1}


def ln_testing_select_kernels(forward="default", backward="default", softmax="default") -> None:
    """Testing hook (include/normfuse_testing.h): plan later calls with the
    default kernels of each shape ("default") or with the bulk-copy ring
    kernels ("ring"), per direction. Process-wide."""
    lib = load_library()
    try:
        codes = [_FAMILY_CODES[v] for v in (forward, backward, softmax)]
    except KeyError as e:
        raise ValueError(f"unknown kernel family {e.args[0]!r}") from None
    st = lib.ln_testing_select_kernels(*codes)
    if st:
        raise NormError(st, "ln_testing_select_kernels")


_PLAN_DIRECTIONS = {"forward": 0, "backward": 1, "softmax": 2, "partials": 3}
_PLAN_FIELDS = ("kind", "group", "n", "block", "grid", "smem")


def ln_testing_plan(direction, rows, hidden, dtype, mode="layernorm", option=False) -> dict:
    """Testing hook (include/normfuse_testing.h): the launch the library
    would plan for this shape on the current device, as a dict of kind,
    group, n, block, grid and smem. ``direction`` is "forward", "backward",
    "softmax" or "partials"; ``option`` a residual (forward) or dbias
    (backward)."""
    lib = load_library()
    try:
        d = _PLAN_DIRECTIONS[direction]
    except KeyError:
        raise ValueError(f"unknown direction {direction!r}") from None
    code = _DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    out = (ctypes.c_int * 6)()
    st = lib.ln_testing_plan(d, int(rows), int(hidden), code, _mode(mode), int(bool(option)), out)
    if st:
        raise NormError(st, "ln_testing_plan")
    return dict(zip(_PLAN_FIELDS, list(out)))


def ln_status_string(status: int) -> str:
    return load_library().ln_status_string(int(status)).decode()


def ln_last_cuda_error() -> int:
    return int(load_library().ln_last_cuda_error())


def ln_device_error(stream=None) -> int:
    """Wait for ``stream`` and return (and clear) the kernels' device error
    bits; 0 means no kernel reported a failed wait."""
    lib = load_library()
    flags = ctypes.c_uint(0)
    st = lib.ln_device_error(_stream(stream), ctypes.byref(flags))
    if st:
        raise NormError(st, "ln_device_error")
    return int(flags.value)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor or None, got {type(t).__name__}")
    if t.numel() and not t.is_cuda:
        raise ValueError("tensors passed to the CUDA library must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr() or None


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _shape(t: torch.Tensor) -> tuple[int, int]:
    if t.dim() < 1:
        raise ValueError("expected at least one dimension (the hidden one)")
    hidden = t.shape[-1]
    return t.numel() // hidden if hidden else 0, hidden


def _mode(mode) -> int:
    try:
        return _MODE_CODES[mode]
    except KeyError:
        raise ValueError(f"unknown mode {mode!r}") from None


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPE_CODES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def ln_fwd(x, bias, residual, gamma, beta, eps, mode, zero_centered_gamma, out_sum, y,
           mean, rstd, amax, stream=None) -> None:
    """Enqueue the fused forward on ``stream`` (default: torch's current stream).

    Tensors: x, residual, out_sum, y are [..., hidden] in one dtype; bias, gamma,
    beta are [hidden]; mean, rstd fp32 [rows]; amax a one-element fp32 tensor.
    Optional ones may be None (see ``ln_fwd`` in include/normfuse.h).
    """
    lib = load_library()
    rows, hidden = _shape(x)
    st = lib.ln_fwd(_ptr(x), _ptr(bias), _ptr(residual), _ptr(gamma), _ptr(beta),
                    float(eps), _mode(mode), int(bool(zero_centered_gamma)), _ptr(out_sum),
                    _ptr(y), _ptr(mean), _ptr(rstd), _ptr(amax), _stream(stream), rows,
                    hidden, _dtype(x))
    if st:
        raise NormError(st, "ln_fwd")


def ln_fwd_ex(x, bias, residual, gamma, beta, eps, mode, zero_centered_gamma, out_sum, y,
              mean, rstd, amax, y_fp8, fp8_scale, stream=None) -> None:
    """``ln_fwd`` plus an FP8 E4M3 copy of y: ``y_fp8`` is a uint8 (or
    torch.float8_e4m3fn) tensor shaped like x, ``fp8_scale`` a one-element fp32
    CUDA tensor; y may be None when y_fp8 is given."""
    lib = load_library()
    rows, hidden = _shape(x)
    st = lib.ln_fwd_ex(_ptr(x), _ptr(bias), _ptr(residual), _ptr(gamma), _ptr(beta),
                       float(eps), _mode(mode), int(bool(zero_centered_gamma)), _ptr(out_sum),
                       _ptr(y), _ptr(mean), _ptr(rstd), _ptr(amax), _ptr(y_fp8),
                       _ptr(fp8_scale), _stream(stream), rows, hidden, _dtype(x))
    if st:
        raise NormError(st, "ln_fwd_ex")


def ln_fwd_from_partials(x, psum, psq, tile_cols, kind, gamma, beta, eps, mode,
                         zero_centered_gamma, y, mean, rstd, amax, stream=None) -> None:
    """Enqueue the normalize step with row statistics combined from per
    column-tile partials: ``psum``/``psq`` are fp32 [rows, ceil(hidden /
    tile_cols)] tensors, ``kind`` "sum_sq" or "sum_m2" (see
    ``ln_fwd_from_partials`` in include/normfuse.h)."""
    lib = load_library()
    rows, hidden = _shape(x)
    n_tiles = psum.shape[-1] if psum is not None else -(-hidden // int(tile_cols))
    try:
        k = _PARTIAL_CODES[kind]
    except KeyError:
        raise ValueError(f"unknown partial kind {kind!r}") from None
    st = lib.ln_fwd_from_partials(_ptr(x), _ptr(psum), _ptr(psq), int(n_tiles), int(tile_cols),
                                  k, _ptr(gamma), _ptr(beta), float(eps), _mode(mode),
                                  int(bool(zero_centered_gamma)), _ptr(y), _ptr(mean),
                                  _ptr(rstd), _ptr(amax), _stream(stream), rows, hidden,
                                  _dtype(x))
    if st:
        raise NormError(st, "ln_fwd_from_partials")


def ln_bwd_workspace_bytes(rows: int, hidden: int, dtype, mode) -> int:
    lib = load_library()
    out = ctypes.c_size_t(0)
    code = _DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    st = lib.ln_bwd_workspace_bytes(int(rows), int(hidden), code, _mode(mode), ctypes.byref(out))
    if st:
        raise NormError(st, "ln_bwd_workspace_bytes")
    return int(out.value)


def ln_bwd(dy, x_sum, gamma, mean, rstd, dx, dgamma, dbeta, stream=None, *, mode="layernorm",
           zero_centered_gamma=False, workspace=None) -> None:
    """Enqueue the fused backward on ``stream``.

    ``workspace`` is a CUDA tensor of at least ``ln_bwd_workspace_bytes`` bytes;
    when None a fresh one is allocated through torch for this call.
    """
    lib = load_library()
    rows, hidden = _shape(dy)
    if workspace is None and rows > 0:
        need = ln_bwd_workspace_bytes(rows, hidden, dy.dtype, mode)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dy.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.ln_bwd(_ptr(dy), _ptr(x_sum), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(dx),
                    _ptr(dgamma), _ptr(dbeta), _stream(stream), rows, hidden, _dtype(dy),
                    _mode(mode), int(bool(zero_centered_gamma)), _ptr(workspace), ws_bytes)
    if st:
        raise NormError(st, "ln_bwd")


def ln_bwd_noalloc(dy, x_sum, gamma, mean, rstd, dx, dgamma, dbeta, stream=None, *,
                   mode="layernorm", zero_centered_gamma=False) -> None:
    """``ln_bwd`` without a workspace: the library's static scratch array holds
    the partials, so neither this call nor the library allocates memory.

    For callers that cannot allocate device memory around the backward
    (see ``ln_bwd_noalloc`` in include/normfuse.h for the size limit and the
    rule that calls overlapping on the GPU race on the shared array).
    """
    lib = load_library()
    rows, hidden = _shape(dy)
    st = lib.ln_bwd_noalloc(_ptr(dy), _ptr(x_sum), _ptr(gamma), _ptr(mean), _ptr(rstd),
                            _ptr(dx), _ptr(dgamma), _ptr(dbeta), _stream(stream), rows, hidden,
                            _dtype(dy), _mode(mode), int(bool(zero_centered_gamma)))
    if st:
        raise NormError(st, "ln_bwd_noalloc")


def ln_bwd_ex(dy, x_sum, gamma, mean, rstd, dx, dgamma, dbeta, dbias, stream=None, *,
              mode="layernorm", zero_centered_gamma=False, workspace=None) -> None:
    """``ln_bwd`` that also writes ``dbias`` ([hidden], the column sum of dx:
    the gradient of the forward's bias; may be None). dgamma, dbeta and dbias
    share one dtype, float32, bfloat16 or float16, taken from ``dgamma``: the
    column totals are rounded once to it."""
    lib = load_library()
    rows, hidden = _shape(dy)
    if workspace is None and rows > 0:
        need = ln_bwd_workspace_bytes(rows, hidden, dy.dtype, mode)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dy.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.ln_bwd_ex(_ptr(dy), _ptr(x_sum), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(dx),
                       _ptr(dgamma), _ptr(dbeta), _ptr(dbias), _stream(stream), rows, hidden,
                       _dtype(dy), _mode(mode), int(bool(zero_centered_gamma)),
                       _ptr(workspace), ws_bytes, _dtype(dgamma))
    if st:
        raise NormError(st, "ln_bwd_ex")


def ln_softmax_fwd(x, y, stream=None) -> None:
    """Enqueue the softmax over the last dimension of the contiguous CUDA
    tensor ``x`` into ``y`` (same shape and dtype; ``y`` may be ``x`` itself)."""
    lib = load_library()
    rows, hidden = _shape(x)
    if y is not x and (y.shape != x.shape or y.dtype != x.dtype):
        raise ValueError("y must have the shape and dtype of x")
    st = lib.ln_softmax_fwd(_ptr(x), _ptr(y), _stream(stream), rows, hidden, _dtype(x))
    if st:
        raise NormError(st, "ln_softmax_fwd")


def softmax_fwd(x, *, out=None, stream=None):
    """Softmax over the last dimension of a contiguous tensor; returns ``y``
    (allocated with torch unless ``out`` is given)."""
    y = torch.empty_like(x) if out is None else out
    ln_softmax_fwd(x, y, stream)
    return y


class Workspace:
    """A reusable backward workspace, grown on demand (allocated through torch)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = torch.empty(0, dtype=torch.uint8, device=self.device)

    def get(self, rows: int, hidden: int, dtype, mode) -> torch.Tensor:
        need = ln_bwd_workspace_bytes(rows, hidden, dtype, mode)
        if self.buf.numel() < need:
            self.buf = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self.buf


def fused_norm_fwd(x, gamma, beta=None, *, bias=None, residual=None, eps=1e-5,
                   mode="layernorm", zero_centered_gamma=False, store_sum=None, amax=False,
                   stream=None):
    """Allocate the outputs with torch and run ``ln_fwd``.

    Returns a dict with ``y``, ``sum`` (or None), ``mean`` (LayerNorm), ``rstd``,
    ``amax`` (or None).
    """
    rows, hidden = _shape(x)
    if store_sum is None:
        store_sum = bias is not None or residual is not None
    rms = _mode(mode) == LN_RMSNORM
    y = torch.empty_like(x)
    out_sum = torch.empty_like(x) if store_sum else None
    mean = None if rms else torch.empty(rows, dtype=torch.float32, device=x.device)
    rstd = torch.empty(rows, dtype=torch.float32, device=x.device)
    am = torch.empty(1, dtype=torch.float32, device=x.device) if amax else None
    ln_fwd(x, bias, residual, gamma, None if rms else beta, eps, mode, zero_centered_gamma,
           out_sum, y, mean, rstd, am, stream)
    return {"y": y, "sum": out_sum, "mean": mean, "rstd": rstd, "amax": am}


def fused_norm_fwd_from_partials(x, psum, psq, tile_cols, gamma, beta=None, *, kind="sum_sq",
                                 eps=1e-5, mode="layernorm", zero_centered_gamma=False,
                                 amax=False, stream=None):
    """Allocate the outputs with torch and run ``ln_fwd_from_partials``;
    returns a dict with ``y``, ``mean`` (LayerNorm), ``rstd``, ``amax``."""
    rows, hidden = _shape(x)
    rms = _mode(mode) == LN_RMSNORM
    y = torch.empty_like(x)
    mean = None if rms else torch.empty(rows, dtype=torch.float32, device=x.device)
    rstd = torch.empty(rows, dtype=torch.float32, device=x.device)
    am = torch.empty(1, dtype=torch.float32, device=x.device) if amax else None
    ln_fwd_from_partials(x, psum, psq, tile_cols, kind, gamma, None if rms else beta, eps, mode,
                         zero_centered_gamma, y, mean, rstd, am, stream)
    return {"y": y, "mean": mean, "rstd": rstd, "amax": am}


def fused_norm_bwd(dy, x_sum, gamma, mean, rstd, *, mode="layernorm", zero_centered_gamma=False,
                   need_dbeta=True, need_dbias=False, grad_dtype=torch.float32,
                   workspace: Workspace | None = None, stream=None):
    """Allocate the outputs with torch and run ``ln_bwd`` (``ln_bwd_ex`` when
    ``need_dbias`` or a ``grad_dtype`` other than float32); returns dx,
    dgamma, dbeta, dbias."""
    rows, hidden = _shape(dy)
    rms = _mode(mode) == LN_RMSNORM
    dx = torch.empty_like(dy)
    g = dict(dtype=grad_dtype, device=dy.device)
    dgamma = torch.empty(hidden, **g)
    dbeta = torch.empty(hidden, **g) if (need_dbeta and not rms) else None
    dbias = torch.empty(hidden, **g) if need_dbias else None
    ws = workspace.get(rows, hidden, dy.dtype, mode) if workspace is not None else None
    if need_dbias or grad_dtype != torch.float32:
        ln_bwd_ex(dy, x_sum, gamma, mean, rstd, dx, dgamma, dbeta, dbias, stream, mode=mode,
                  zero_centered_gamma=zero_centered_gamma, workspace=ws)
    else:
        ln_bwd(dy, x_sum, gamma, mean, rstd, dx, dgamma, dbeta, stream, mode=mode,
               zero_centered_gamma=zero_centered_gamma, workspace=ws)
    return {"dx": dx, "dgamma": dgamma, "dbeta": dbeta, "dbias": dbias}
