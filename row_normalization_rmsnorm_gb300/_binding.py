"""ctypes binding of libgb300norm.so (the C ABI in include/gb300norm.h).

Argument marshalling only: every function below takes torch tensors that
already live on the current CUDA device, passes their data pointers, row
strides, shapes and dtype codes to the C entry point of the same name and
raises NormError on a non-zero status.  Nothing is computed here and there is
no CPU path: a CPU tensor, or a missing library, is an error.
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


def _dev(t, name, dims=None):
    """Data pointer of a CUDA tensor (or None), checked for device and layout."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    st = t.stride()
    nd = len(st)
    if dims is not None and nd != dims:
        raise ValueError(f"{name} must be {dims}-D, got shape {tuple(t.shape)}")
    if nd == 2 and st[1] != 1 and t.shape[1] > 1:
        raise ValueError(f"{name} rows must be contiguous (stride(1) == 1)")
    if nd == 1 and st[0] != 1 and t.numel() > 1:
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr() or None


def _rs(t):
    return t.stride(0) if (t is not None and t.dim() == 2) else 0


def _ptr(t):
    return None if t is None else (t.data_ptr() or None)


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


def norm_rms_fwd(x, w, y, rstd=None, offset=0.0, eps=1e-6, stream=None):
    """y = RMSNorm(x) with scale (w + offset); rstd (FP32, [M]) optional."""
    M, N = x.shape
    rc = lib.norm_rms_fwd(_dev(x, "x", 2), _rs(x), _dev(w, "w", 1), _dev(y, "y", 2), _rs(y),
                          _dev(rstd, "rstd", 1), M, N, float(offset), float(eps),
                          DTYPE_CODE[x.dtype], DTYPE_CODE[w.dtype], _stream(stream, x))
    _check("norm_rms_fwd", rc)


def norm_rms_bwd(dy, x, w, rstd, dx, dw=None, workspace=None, offset=0.0, eps=1e-6, stream=None):
    """dx (and dw unless None = frozen) of RMSNorm; rstd None = recompute."""
    M, N = x.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.norm_rms_bwd(_dev(dy, "dy", 2), _rs(dy), _dev(x, "x", 2), _rs(x), _dev(w, "w", 1),
                          _dev(rstd, "rstd", 1), _dev(dx, "dx", 2), _rs(dx),
                          _dev(dw, "dw", 1), DTYPE_CODE[dw.dtype] if dw is not None else NORM_F32,
                          _dev(workspace, "workspace"), ws_bytes, M, N, float(offset), float(eps),
                          DTYPE_CODE[x.dtype], DTYPE_CODE[w.dtype], _stream(stream, x))
    _check("norm_rms_bwd", rc)


def norm_rms_bwd_noalloc(dy, x, w, rstd, dx, dw=None, offset=0.0, eps=1e-6, stream=None):
    """norm_rms_bwd without a workspace: the dW partial sums use the
    library's fixed scratch (for callers that cannot allocate)."""
    M, N = x.shape
    rc = lib.norm_rms_bwd_noalloc(_dev(dy, "dy", 2), _rs(dy), _dev(x, "x", 2), _rs(x), _dev(w, "w", 1),
                                  _dev(rstd, "rstd", 1), _dev(dx, "dx", 2), _rs(dx), _dev(dw, "dw", 1),
                                  DTYPE_CODE[dw.dtype] if dw is not None else NORM_F32, M, N, float(offset),
                                  float(eps), DTYPE_CODE[x.dtype], DTYPE_CODE[w.dtype], _stream(stream, x))
    _check("norm_rms_bwd_noalloc", rc)


def norm_ln_fwd(x, w, b, y, mean=None, rstd=None, offset=0.0, eps=1e-6, stream=None):
    """y = LayerNorm(x) with scale (w + offset) and bias b (None = no bias)."""
    M, N = x.shape
    rc = lib.norm_ln_fwd(_dev(x, "x", 2), _rs(x), _dev(w, "w", 1), _dev(b, "b", 1), _dev(y, "y", 2), _rs(y),
                         _dev(mean, "mean", 1), _dev(rstd, "rstd", 1), M, N, float(offset), float(eps),
                         DTYPE_CODE[x.dtype], DTYPE_CODE[w.dtype], _stream(stream, x))
    _check("norm_ln_fwd", rc)


def norm_ln_bwd(dy, x, w, mean, rstd, dx, dw=None, db=None, workspace=None, offset=0.0, eps=1e-6,
                stream=None):
    """dx, and dw / db unless None (frozen), of LayerNorm."""
    M, N = x.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    gd = dw if dw is not None else db
    rc = lib.norm_ln_bwd(_dev(dy, "dy", 2), _rs(dy), _dev(x, "x", 2), _rs(x), _dev(w, "w", 1),
                         _dev(mean, "mean", 1), _dev(rstd, "rstd", 1), _dev(dx, "dx", 2), _rs(dx),
                         _dev(dw, "dw", 1), _dev(db, "db", 1),
                         DTYPE_CODE[gd.dtype] if gd is not None else NORM_F32,
                         _dev(workspace, "workspace"), ws_bytes, M, N, float(offset), float(eps),
                         DTYPE_CODE[x.dtype], DTYPE_CODE[w.dtype], _stream(stream, x))
    _check("norm_ln_bwd", rc)


def norm_fused_add_rms_fwd(x, residual, w, y, h_out, rstd=None, offset=0.0, eps=1e-6, stream=None):
    """h_out = x + residual (rounded), y = RMSNorm(h) with scale (w + offset)."""
    M, N = x.shape
    rc = lib.norm_fused_add_rms_fwd(_dev(x, "x", 2), _rs(x), _dev(residual, "residual", 2), _rs(residual),
                                    _dev(w, "w", 1), _dev(y, "y", 2), _rs(y), _dev(h_out, "h_out", 2),
                                    _rs(h_out), _dev(rstd, "rstd", 1), M, N, float(offset), float(eps),
                                    DTYPE_CODE[x.dtype], DTYPE_CODE[w.dtype], _stream(stream, x))
    _check("norm_fused_add_rms_fwd", rc)


def norm_fused_add_rms_bwd(dy, dh_out, h, w, rstd, dx, dw=None, workspace=None, offset=0.0, eps=1e-6,
                           stream=None):
    """dx (= d residual) and dw unless None, of FusedAddRMSNorm at saved h."""
    M, N = h.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.norm_fused_add_rms_bwd(_dev(dy, "dy", 2), _rs(dy), _dev(dh_out, "dh_out", 2), _rs(dh_out),
                                    _dev(h, "h", 2), _rs(h), _dev(w, "w", 1), _dev(rstd, "rstd", 1),
                                    _dev(dx, "dx", 2), _rs(dx), _dev(dw, "dw", 1),
                                    DTYPE_CODE[dw.dtype] if dw is not None else NORM_F32,
                                    _dev(workspace, "workspace"), ws_bytes, M, N, float(offset), float(eps),
                                    DTYPE_CODE[h.dtype], DTYPE_CODE[w.dtype], _stream(stream, h))
    _check("norm_fused_add_rms_bwd", rc)
