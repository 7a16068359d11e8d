"""FP64 CPU oracle for row-wise RMSNorm, LayerNorm and FusedAddRMSNorm.

TEST INFRASTRUCTURE ONLY.  The product library never imports, links or runs
anything in this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA path.

The arithmetic lives in ``norm_oracle.c`` (plain C, FP64, one row after
another).  This module compiles it with gcc, loads it with ctypes and wraps
each entry point for dense ``numpy.float64`` arrays.  Every function returns
FP64 results; ``round_to`` rounds them once, directly from FP64, to a storage
type (round to nearest, ties to even).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(library special cases, finite differences, closed forms, per-row invariants,
the pages' worked BF16 example and a brute-force rounding check).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "norm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libnormoracle.so")

DTYPE_CODES = {"float32": 0, "float16": 1, "bfloat16": 2}

_lib = None


def build(force: bool = False) -> str:
    """Compile norm_oracle.c into libnormoracle.so (gcc, FP contraction off)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I = ctypes.c_int64
    D = ctypes.c_double
    lib.oracle_rms_fwd.argtypes = [I, I, P, P, D, D, P, P]
    lib.oracle_rms_bwd.argtypes = [I, I, P, P, P, D, D, P, P, P, P]
    lib.oracle_ln_fwd.argtypes = [I, I, P, P, P, D, D, P, P, P, P]
    lib.oracle_ln_bwd.argtypes = [I, I, P, P, P, D, D, P, P, P, P, P, P]
    lib.oracle_fused_add_rms_fwd.argtypes = [I, I, P, P, P, D, D, P, P, P]
    lib.oracle_fused_add_rms_bwd.argtypes = [I, I, P, P, P, P, D, D, P, P, P, P]
    lib.oracle_round_array.argtypes = [P, I, ctypes.c_int, P]
    lib.oracle_round_bf16.argtypes = [D]
    lib.oracle_round_bf16.restype = ctypes.c_uint16
    lib.oracle_round_f16.argtypes = [D]
    lib.oracle_round_f16.restype = ctypes.c_uint16
    for f in (lib.oracle_rms_fwd, lib.oracle_rms_bwd, lib.oracle_ln_fwd,
              lib.oracle_ln_bwd, lib.oracle_fused_add_rms_fwd,
              lib.oracle_fused_add_rms_bwd, lib.oracle_round_array):
        f.restype = None
    _lib = lib
    return lib


def _in(a, shape=None):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None:
        a = a.reshape(shape)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _opt(flag, shape):
    return np.empty(shape, dtype=np.float64) if flag else None


def rms_fwd(x, w, offset=0.0, eps=1e-6):
    """RMSNorm forward. Returns (y, rstd)."""
    lib = _load()
    x = _in(x)
    M, N = x.shape
    w = _in(w, (N,))
    y = np.empty((M, N))
    rstd = np.empty(M)
    lib.oracle_rms_fwd(M, N, _ptr(x), _ptr(w), offset, eps, _ptr(y), _ptr(rstd))
    return y, rstd


def rms_bwd(x, dy, w, offset=0.0, eps=1e-6, compute_dw=True, with_scale=False, rstd=None):
    """RMSNorm backward. rstd: the forward's saved statistic (None = recompute).
    Returns (dx, dw or None, dx_scale or None)."""
    lib = _load()
    x = _in(x)
    M, N = x.shape
    dy = _in(dy, (M, N))
    w = _in(w, (N,))
    rs = None if rstd is None else _in(rstd, (M,))
    dx = np.empty((M, N))
    dw = _opt(compute_dw, N)
    sc = _opt(with_scale, (M, N))
    lib.oracle_rms_bwd(M, N, _ptr(x), _ptr(dy), _ptr(w), offset, eps,
                       _ptr(dx), _ptr(dw), _ptr(sc), _ptr(rs))
    return dx, dw, sc


def ln_fwd(x, w, b=None, offset=0.0, eps=1e-6, with_scale=False):
    """LayerNorm forward. Returns (y, mean, rstd, y_scale or None)."""
    lib = _load()
    x = _in(x)
    M, N = x.shape
    w = _in(w, (N,))
    b = None if b is None else _in(b, (N,))
    y = np.empty((M, N))
    mean = np.empty(M)
    rstd = np.empty(M)
    sc = _opt(with_scale, (M, N))
    lib.oracle_ln_fwd(M, N, _ptr(x), _ptr(w), _ptr(b), offset, eps, _ptr(y),
                      _ptr(mean), _ptr(rstd), _ptr(sc))
    return y, mean, rstd, sc


def ln_bwd(x, dy, w, offset=0.0, eps=1e-6, compute_dw=True, compute_db=True,
           with_scale=False, mean=None, rstd=None):
    """LayerNorm backward. mean / rstd: the forward's saved statistics (both
    or neither; None = recompute). Returns (dx, dw or None, db or None,
    dx_scale or None)."""
    lib = _load()
    x = _in(x)
    M, N = x.shape
    dy = _in(dy, (M, N))
    w = _in(w, (N,))
    if (mean is None) != (rstd is None):
        raise ValueError("mean and rstd go together")
    mu = None if mean is None else _in(mean, (M,))
    rs = None if rstd is None else _in(rstd, (M,))
    dx = np.empty((M, N))
    dw = _opt(compute_dw, N)
    db = _opt(compute_db, N)
    sc = _opt(with_scale, (M, N))
    lib.oracle_ln_bwd(M, N, _ptr(x), _ptr(dy), _ptr(w), offset, eps, _ptr(dx),
                      _ptr(dw), _ptr(db), _ptr(sc), _ptr(mu), _ptr(rs))
    return dx, dw, db, sc


def fused_add_rms_fwd(x, residual, w, offset=0.0, eps=1e-6):
    """FusedAddRMSNorm forward. Returns (y, h, rstd) with h = x + residual exact."""
    lib = _load()
    x = _in(x)
    M, N = x.shape
    r = _in(residual, (M, N))
    w = _in(w, (N,))
    y = np.empty((M, N))
    h = np.empty((M, N))
    rstd = np.empty(M)
    lib.oracle_fused_add_rms_fwd(M, N, _ptr(x), _ptr(r), _ptr(w), offset, eps,
                                 _ptr(y), _ptr(h), _ptr(rstd))
    return y, h, rstd


def fused_add_rms_bwd(h, dy, w, dh_out=None, offset=0.0, eps=1e-6,
                      compute_dw=True, with_scale=False, rstd=None):
    """FusedAddRMSNorm backward from the saved rows h (as stored by the
    forward) and the forward's rstd (None = recompute from h).

    Returns (dx, dw or None, dx_scale or None); dx is also the residual
    gradient.
    """
    lib = _load()
    h = _in(h)
    M, N = h.shape
    dy = _in(dy, (M, N))
    w = _in(w, (N,))
    dho = None if dh_out is None else _in(dh_out, (M, N))
    rs = None if rstd is None else _in(rstd, (M,))
    dx = np.empty((M, N))
    dw = _opt(compute_dw, N)
    sc = _opt(with_scale, (M, N))
    lib.oracle_fused_add_rms_bwd(M, N, _ptr(h), _ptr(dy), _ptr(dho), _ptr(w),
                                 offset, eps, _ptr(dx), _ptr(dw), _ptr(sc), _ptr(rs))
    return dx, dw, sc


def round_to(a, dtype: str):
    """Round FP64 values once to `dtype` ('float32' | 'float16' | 'bfloat16').

    float32 returns a float32 array; float16 / bfloat16 return uint16 arrays
    of bit patterns (view them with torch's .view(torch.bfloat16) etc.).
    """
    lib = _load()
    a = np.ascontiguousarray(a, dtype=np.float64)
    code = DTYPE_CODES[dtype]
    out = np.empty(a.shape, dtype=np.float32 if code == 0 else np.uint16)
    lib.oracle_round_array(_ptr(a), a.size, code, out.ctypes.data_as(ctypes.c_void_p))
    return out


def round_bf16_bits(v: float) -> int:
    return int(_load().oracle_round_bf16(float(v)))


def round_f16_bits(v: float) -> int:
    return int(_load().oracle_round_f16(float(v)))
