"""ctypes binding of libgb300norm.so (the C ABI in include/gb300norm.h).

Argument marshalling only: every function below takes torch tensors on one
CUDA device, passes their data pointers, row strides, shapes and dtype codes
to the C entry point of the same name (with that device current) and raises
NormError on a non-zero status.  Nothing is computed here and there is no
CPU path: a CPU tensor, or a missing library, is an error.

The C ABI sees only pointers, so the extent of every buffer is checked here
before the call: each 2-D tensor must be (M, N) in the activation dtype with
contiguous rows, w / b / dW / dB must hold N elements, rstd / mean at least
M FP32 values, and every tensor must sit on x's device.  Shape and dtype
errors raise ValueError (before any device check), a CPU tensor TypeError.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgb300norm.so")

NORM_F32, NORM_F16, NORM_BF16 = 0, 1, 2
DTYPE_CODE = {torch.float32: NORM_F32, torch.float16: NORM_F16, torch.bfloat16: NORM_BF16}
CODE_DTYPE = {v: k for k, v in DTYPE_CODE.items()}

# status codes (include/gb300norm.h)
NORM_OK = 0
NORM_ERR_NULL = 1
NORM_ERR_SHAPE = 2
NORM_ERR_STRIDE = 3
NORM_ERR_DTYPE = 4
NORM_ERR_WORKSPACE = 5
NORM_ERR_ALIGN = 6
NORM_ERR_VALUE = 7
NORM_ERR_ALIAS = 8
NORM_ERR_CUDA = 9
NORM_ERR_ARG = 10
NORM_ERR_TOO_LARGE = 11

# Every entry point the header declares, with its ctypes signature.
_P, _I64, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "norm_status_str": ([_I], ctypes.c_char_p),
    "norm_version": ([], _I),
    "norm_bwd_workspace_bytes": ([_I64, _I64, _I, _I, ctypes.POINTER(_SZ)], _I),
    "norm_rms_fwd": ([_P, _I64, _P, _P, _I64, _P, _I64, _I64, _F, _F, _I, _I, _P], _I),
    "norm_rms_bwd": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I, _P, _SZ, _I64, _I64, _F, _F, _I, _I, _P], _I),
    "norm_ln_fwd": ([_P, _I64, _P, _P, _P, _I64, _P, _P, _I64, _I64, _F, _F, _I, _I, _P], _I),
    "norm_ln_bwd": ([_P, _I64, _P, _I64, _P, _P, _P, _P, _I64, _P, _P, _I, _P, _SZ, _I64, _I64, _F, _F, _I, _I,
                     _P], _I),
    "norm_fused_add_rms_fwd": ([_P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _P, _I64, _I64, _F, _F, _I, _I, _P],
                               _I),
    "norm_fused_add_rms_bwd": ([_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I, _P, _SZ, _I64, _I64, _F,
                                _F, _I, _I, _P], _I),
    "norm_device_status": ([_I, ctypes.POINTER(_I)], _I),
    "norm_debug_set_path": ([_I], _I),
    "norm_debug_tune": ([_I, _I], _I),
    "norm_last_cuda_error": ([], _I),
    "norm_noalloc_scratch_bytes": ([], _SZ),
    "norm_rms_bwd_noalloc": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I, _I64, _I64, _F, _F, _I, _I, _P], _I),
    "norm_cuda_error_string": ([_I], ctypes.c_char_p),
    "norm_sum_ranks": ([_P, _I64, _I64, _P, _I, _P], _I),
    "norm_debug_launches": ([_I], _I64),
}


class NormError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn}: status {status} ({status_str(status)})"
        if status == NORM_ERR_CUDA:
            code = lib.norm_last_cuda_error()
            msg += f"; CUDA error {code}: {lib.norm_cuda_error_string(code).decode()}"
        super().__init__(msg)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(nvcc, sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in SIGNATURES.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


lib = _load()


def status_str(status: int) -> str:
    return lib.norm_status_str(int(status)).decode()


def _check(fn: str, rc: int):
    if rc != NORM_OK:
        raise NormError(fn, rc)


# The current stream's raw handle without building a torch.cuda.Stream object
# on every call (that alone cost more than the rest of a small call).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, like=None):
    """Raw cudaStream_t (an int) for the C ABI: `stream`, else the current
    stream of `like`'s device (else of the current device)."""
    if stream is None:
        if _raw_stream is not None:
            dev = like.get_device() if like is not None else torch.cuda.current_device()
            return _raw_stream(dev)
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _tensor(t, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    return t


def _mat(t, name, M, N, dtype, required=True):
    """Check a 2-D row tensor: shape (M, N), the activation dtype, rows
    contiguous.  Runs before any device check, so a shape error is reported
    as such whatever the tensor's device."""
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return
    _tensor(t, name)
    if t.dim() != 2 or tuple(t.shape) != (M, N):
        raise ValueError(f"{name} must have shape ({M}, {N}), got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if M > 0 and N > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous (stride(1) == 1)")


def _vec(t, name, n, dtypes, at_least=False, required=True):
    """Check a 1-D contiguous vector of n elements (at least n when
    `at_least`) whose dtype is one of `dtypes`."""
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return
    _tensor(t, name)
    if t.dim() != 1:
        raise ValueError(f"{name} must be 1-D, got shape {tuple(t.shape)}")
    if (t.numel() < n) if at_least else (t.numel() != n):
        raise ValueError(f"{name} must have {'at least ' if at_least else ''}{n} elements, got {t.numel()}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must be one of {[str(d) for d in dtypes]}, got {t.dtype}")
    if t.numel() > 1 and t.stride(0) != 1:
        raise ValueError(f"{name} must be contiguous")


def _act_dtype(x, name="x"):
    _tensor(x, name)
    if x.dim() != 2:
        raise ValueError(f"{name} must be 2-D [M, N], got shape {tuple(x.shape)}")
    if x.dtype not in DTYPE_CODE:
        raise ValueError(f"{name} dtype {x.dtype} is not supported")
    return x.dtype


def _weight(w, N):
    _tensor(w, "w")
    _vec(w, "w", N, tuple(DTYPE_CODE))
    return w.dtype


def _grad_dtype(w_dtype, *grads):
    """dtype code of the dW / dB outputs: FP32 or the weight's dtype, the
    same for every gradient given."""
    given = [(n, t) for n, t in grads if t is not None]
    if not given:
        return NORM_F32
    dt = given[0][1].dtype
    if dt not in (torch.float32, w_dtype):
        raise ValueError(f"{given[0][0]} must be float32 or the weight dtype {w_dtype}, got {dt}")
    for n, t in given[1:]:
        if t.dtype != dt:
            raise ValueError(f"{n} must have the same dtype as {given[0][0]} ({dt}), got {t.dtype}")
    return DTYPE_CODE[dt]


def _device(x, *others):
    """Index of the CUDA device every tensor lives on (x's), or an error."""
    if not x.is_cuda:
        raise TypeError("x must be a CUDA tensor (this library has no CPU path)")
    dev = x.get_device()
    for name, t in others:
        if t is None:
            continue
        if not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor (this library has no CPU path)")
        if t.get_device() != dev:
            raise ValueError(f"{name} is on cuda:{t.get_device()}, x on cuda:{dev}")
    return dev


def _on(dev, fn):
    """Run fn with `dev` as the current device: the C ABI takes its device
    (launch shapes, status word) from the current device."""
    if dev == torch.cuda.current_device():
        return fn()
    with torch.cuda.device(dev):
        return fn()


def _rs(t):
    return t.stride(0) if (t is not None and t.dim() == 2) else 0


def _ptr(t):
    return None if t is None else (t.data_ptr() or None)


def _ws(workspace):
    if workspace is None:
        return None, 0
    _tensor(workspace, "workspace")
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    return workspace.data_ptr() or None, workspace.numel() * workspace.element_size()


def norm_bwd_workspace_bytes(M: int, N: int, has_dw: bool, has_db: bool = False) -> int:
    out = ctypes.c_size_t(0)
    _check("norm_bwd_workspace_bytes", lib.norm_bwd_workspace_bytes(M, N, int(has_dw), int(has_db),
                                                                    ctypes.byref(out)))
    return out.value


def norm_device_status(reset: bool = False) -> int:
    v = ctypes.c_int(0)
    _check("norm_device_status", lib.norm_device_status(int(reset), ctypes.byref(v)))
    return v.value


def norm_debug_set_path(mode: int):
    _check("norm_debug_set_path", lib.norm_debug_set_path(int(mode)))


def norm_debug_tune(key: int, value: int):
    _check("norm_debug_tune", lib.norm_debug_tune(int(key), int(value)))


def norm_debug_launches(reset: bool = False) -> int:
    """Kernels this library has launched since load or the last reset."""
    return int(lib.norm_debug_launches(int(reset)))


_F32 = (torch.float32,)


def norm_sum_ranks(parts, out, stream=None):
    """out = the rows of parts (FP32, [world, N], one per rank) added in rank
    order in FP32 and converted once to out's dtype (FP32, FP16 or BF16, N
    elements)."""
    _tensor(parts, "parts")
    if parts.dim() != 2 or parts.shape[0] < 1 or parts.shape[1] < 1:
        raise ValueError(f"parts must be 2-D [world, N] with world, N >= 1, got shape {tuple(parts.shape)}")
    if parts.dtype != torch.float32:
        raise ValueError(f"parts must be float32, got {parts.dtype}")
    if not parts.is_contiguous():
        raise ValueError("parts must be contiguous")
    world, N = parts.shape
    _vec(out, "out", N, tuple(DTYPE_CODE))
    dev = _device(parts, ("out", out))
    _on(dev, lambda: _check("norm_sum_ranks", lib.norm_sum_ranks(
        _ptr(parts), world, N, _ptr(out), DTYPE_CODE[out.dtype], _stream(stream, parts))))


def norm_rms_fwd(x, w, y, rstd=None, offset=0.0, eps=1e-6, stream=None):
    """y = RMSNorm(x) with scale (w + offset); rstd (FP32, [M]) optional."""
    dt = _act_dtype(x)
    M, N = x.shape
    wdt = _weight(w, N)
    _mat(y, "y", M, N, dt)
    _vec(rstd, "rstd", M, _F32, at_least=True, required=False)
    dev = _device(x, ("w", w), ("y", y), ("rstd", rstd))
    _on(dev, lambda: _check("norm_rms_fwd", lib.norm_rms_fwd(
        _ptr(x), _rs(x), _ptr(w), _ptr(y), _rs(y), _ptr(rstd), M, N, float(offset), float(eps),
        DTYPE_CODE[dt], DTYPE_CODE[wdt], _stream(stream, x))))


def _rms_bwd_checks(dy, x, w, rstd, dx, dw):
    dt = _act_dtype(x)
    M, N = x.shape
    wdt = _weight(w, N)
    _mat(dy, "dy", M, N, dt)
    _mat(dx, "dx", M, N, dt)
    _vec(rstd, "rstd", M, _F32, at_least=True, required=False)
    _vec(dw, "dw", N, (torch.float32, wdt), required=False)
    dwt = _grad_dtype(wdt, ("dw", dw))
    dev = _device(x, ("dy", dy), ("w", w), ("rstd", rstd), ("dx", dx), ("dw", dw))
    return dt, wdt, dwt, dev


def norm_rms_bwd(dy, x, w, rstd, dx, dw=None, workspace=None, offset=0.0, eps=1e-6, stream=None):
    """dx (and dw unless None = frozen) of RMSNorm; rstd None = recompute."""
    dt, wdt, dwt, dev = _rms_bwd_checks(dy, x, w, rstd, dx, dw)
    M, N = x.shape
    _device(x, ("workspace", workspace))
    wsp, wsb = _ws(workspace)
    _on(dev, lambda: _check("norm_rms_bwd", lib.norm_rms_bwd(
        _ptr(dy), _rs(dy), _ptr(x), _rs(x), _ptr(w), _ptr(rstd), _ptr(dx), _rs(dx), _ptr(dw), dwt, wsp, wsb,
        M, N, float(offset), float(eps), DTYPE_CODE[dt], DTYPE_CODE[wdt], _stream(stream, x))))


def norm_rms_bwd_noalloc(dy, x, w, rstd, dx, dw=None, offset=0.0, eps=1e-6, stream=None):
    """norm_rms_bwd without a workspace: the dW partial sums use the
    library's fixed scratch (for callers that cannot allocate)."""
    dt, wdt, dwt, dev = _rms_bwd_checks(dy, x, w, rstd, dx, dw)
    M, N = x.shape
    _on(dev, lambda: _check("norm_rms_bwd_noalloc", lib.norm_rms_bwd_noalloc(
        _ptr(dy), _rs(dy), _ptr(x), _rs(x), _ptr(w), _ptr(rstd), _ptr(dx), _rs(dx), _ptr(dw), dwt, M, N,
        float(offset), float(eps), DTYPE_CODE[dt], DTYPE_CODE[wdt], _stream(stream, x))))


def norm_ln_fwd(x, w, b, y, mean=None, rstd=None, offset=0.0, eps=1e-6, stream=None):
    """y = LayerNorm(x) with scale (w + offset) and bias b (None = no bias)."""
    dt = _act_dtype(x)
    M, N = x.shape
    wdt = _weight(w, N)
    _vec(b, "b", N, (wdt,), required=False)
    _mat(y, "y", M, N, dt)
    _vec(mean, "mean", M, _F32, at_least=True, required=False)
    _vec(rstd, "rstd", M, _F32, at_least=True, required=False)
    dev = _device(x, ("w", w), ("b", b), ("y", y), ("mean", mean), ("rstd", rstd))
    _on(dev, lambda: _check("norm_ln_fwd", lib.norm_ln_fwd(
        _ptr(x), _rs(x), _ptr(w), _ptr(b), _ptr(y), _rs(y), _ptr(mean), _ptr(rstd), M, N, float(offset),
        float(eps), DTYPE_CODE[dt], DTYPE_CODE[wdt], _stream(stream, x))))


def norm_ln_bwd(dy, x, w, mean, rstd, dx, dw=None, db=None, workspace=None, offset=0.0, eps=1e-6,
                stream=None):
    """dx, and dw / db unless None (frozen), of LayerNorm."""
    dt = _act_dtype(x)
    M, N = x.shape
    wdt = _weight(w, N)
    _mat(dy, "dy", M, N, dt)
    _mat(dx, "dx", M, N, dt)
    _vec(mean, "mean", M, _F32, at_least=True, required=False)
    _vec(rstd, "rstd", M, _F32, at_least=True, required=False)
    _vec(dw, "dw", N, (torch.float32, wdt), required=False)
    _vec(db, "db", N, (torch.float32, wdt), required=False)
    dwt = _grad_dtype(wdt, ("dw", dw), ("db", db))
    dev = _device(x, ("dy", dy), ("w", w), ("mean", mean), ("rstd", rstd), ("dx", dx), ("dw", dw), ("db", db),
                  ("workspace", workspace))
    wsp, wsb = _ws(workspace)
    _on(dev, lambda: _check("norm_ln_bwd", lib.norm_ln_bwd(
        _ptr(dy), _rs(dy), _ptr(x), _rs(x), _ptr(w), _ptr(mean), _ptr(rstd), _ptr(dx), _rs(dx), _ptr(dw),
        _ptr(db), dwt, wsp, wsb, M, N, float(offset), float(eps), DTYPE_CODE[dt], DTYPE_CODE[wdt],
        _stream(stream, x))))


def norm_fused_add_rms_fwd(x, residual, w, y, h_out, rstd=None, offset=0.0, eps=1e-6, stream=None):
    """h_out = x + residual (rounded), y = RMSNorm(h) with scale (w + offset)."""
    dt = _act_dtype(x)
    M, N = x.shape
    wdt = _weight(w, N)
    _mat(residual, "residual", M, N, dt)
    _mat(y, "y", M, N, dt)
    _mat(h_out, "h_out", M, N, dt)
    _vec(rstd, "rstd", M, _F32, at_least=True, required=False)
    dev = _device(x, ("residual", residual), ("w", w), ("y", y), ("h_out", h_out), ("rstd", rstd))
    _on(dev, lambda: _check("norm_fused_add_rms_fwd", lib.norm_fused_add_rms_fwd(
        _ptr(x), _rs(x), _ptr(residual), _rs(residual), _ptr(w), _ptr(y), _rs(y), _ptr(h_out), _rs(h_out),
        _ptr(rstd), M, N, float(offset), float(eps), DTYPE_CODE[dt], DTYPE_CODE[wdt], _stream(stream, x))))


def norm_fused_add_rms_bwd(dy, dh_out, h, w, rstd, dx, dw=None, workspace=None, offset=0.0, eps=1e-6,
                           stream=None):
    """dx (= d residual) and dw unless None, of FusedAddRMSNorm at saved h."""
    dt = _act_dtype(h, "h")
    M, N = h.shape
    wdt = _weight(w, N)
    _mat(dy, "dy", M, N, dt)
    _mat(dh_out, "dh_out", M, N, dt, required=False)
    _mat(dx, "dx", M, N, dt)
    _vec(rstd, "rstd", M, _F32, at_least=True, required=False)
    _vec(dw, "dw", N, (torch.float32, wdt), required=False)
    dwt = _grad_dtype(wdt, ("dw", dw))
    dev = _device(h, ("dy", dy), ("dh_out", dh_out), ("w", w), ("rstd", rstd), ("dx", dx), ("dw", dw),
                  ("workspace", workspace))
    wsp, wsb = _ws(workspace)
    _on(dev, lambda: _check("norm_fused_add_rms_bwd", lib.norm_fused_add_rms_bwd(
        _ptr(dy), _rs(dy), _ptr(dh_out), _rs(dh_out), _ptr(h), _rs(h), _ptr(w), _ptr(rstd), _ptr(dx), _rs(dx),
        _ptr(dw), dwt, wsp, wsb, M, N, float(offset), float(eps), DTYPE_CODE[dt], DTYPE_CODE[wdt],
        _stream(stream, h))))
