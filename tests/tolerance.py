"""Parity criteria between the CUDA path and the FP64 oracle.

Tolerances follow the stated bar: FP32 outputs within a relative error of
1e-5; BF16 / FP16 outputs within one unit in the last place of the FP64
oracle rounded (once, directly) to that type; dW / dB within a relative L2
error of 1e-4 when reduced to FP32, and within one ulp of the rounded oracle
when stored in BF16 / FP16.

Where an output is a difference of terms much larger than itself (an input
gradient, a LayerNorm output), FP32 rounding of those terms can exceed one ulp
of the tiny result.  Each check therefore also accepts
``|gpu - ref| <= floor * scale``, where ``scale`` is the magnitude of the
summed terms (from the oracle's *_scale outputs) and ``floor`` is 2^-17 for
FP32 (below the 1e-5 relative bar, measured against those terms) and 2^-16
for BF16 / FP16 outputs; the number of elements that pass only through this
clause is reported and bounded (1 % of the elements).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

FLOOR = {"float32": 2.0 ** -17, "float16": 2.0 ** -16, "bfloat16": 2.0 ** -16}
REL_F32 = 1e-5
DW_REL_L2 = 1e-4

# Every check() report of this test session, printed as a summary at the end
# of the run (tests/conftest.py): how many elements of each output passed
# only through the floor clause.
REPORTS: list = []

_NAMES = {torch.float32: "float32", torch.float16: "float16", torch.bfloat16: "bfloat16"}


def dtype_name(t):
    return _NAMES[t if isinstance(t, torch.dtype) else t.dtype]


def rounded(ref: np.ndarray, name: str) -> np.ndarray:
    """FP64 oracle values rounded once to `name`, returned as float64."""
    r = oracle.round_to(ref, name)
    if name == "float32":
        return r.astype(np.float64)
    tdt = torch.bfloat16 if name == "bfloat16" else torch.float16
    return torch.from_numpy(r.view(np.int16)).view(tdt).double().numpy()


def ulp(v: np.ndarray, name: str) -> np.ndarray:
    """Spacing of the `name` grid at |v| (the gap to the next larger magnitude)."""
    mbits, emin = {"bfloat16": (7, -126), "float16": (10, -14), "float32": (23, -126)}[name]
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, emin), emin)
    return np.exp2(e - mbits)


class Report(dict):
    def __str__(self):
        return ", ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}" for k, v in self.items())


def check(gpu, ref, name_out: str, scale=None, label: str = "", max_floor_frac=1e-2, floor=None):
    """Element-wise parity of `gpu` (torch tensor, any device) against `ref`.

    Returns a Report; raises AssertionError listing the worst elements.
    """
    g = gpu.detach().double().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (label, g.shape, ref.shape)
    fin = np.isfinite(ref)
    # non-finite oracle values must be matched exactly (inf sign / NaN)
    if not fin.all():
        assert np.array_equal(np.isnan(g[~fin]), np.isnan(ref[~fin])), label
        assert np.array_equal(g[~fin][~np.isnan(ref[~fin])], ref[~fin][~np.isnan(ref[~fin])]), label
    g, r, s = g[fin], ref[fin], (None if scale is None else np.asarray(scale, np.float64)[fin])
    err = np.abs(g - r)
    if name_out == "float32":
        ok_main = err <= REL_F32 * np.abs(r)
    else:
        rr = rounded(r, name_out)
        ok_main = np.abs(g - rr) <= ulp(rr, name_out)
    ok = ok_main.copy()
    n_floor = 0
    if s is not None:
        ok_floor = err <= (FLOOR[name_out] if floor is None else floor) * s
        n_floor = int((ok_floor & ~ok_main).sum())
        ok |= ok_floor
    rep = Report(label=label, n=int(r.size), n_floor_only=n_floor,
                 max_abs=float(err.max()) if err.size else 0.0,
                 rel_l2=float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)))
    REPORTS.append(rep)
    if not ok.all():
        bad = np.flatnonzero(~ok)
        worst = bad[np.argsort(-err[bad])[:8]]
        lines = [f"  idx={i} gpu={g[i]!r} ref={r[i]!r} err={err[i]:.3g}"
                 + ("" if s is None else f" scale={s[i]:.3g}") for i in worst]
        raise AssertionError(f"{label}: {bad.size} of {r.size} elements out of tolerance ({rep})\n"
                             + "\n".join(lines))
    # a statistical sanity bound for large arrays; tiny ones (a two-element
    # LayerNorm row has dx = 0 up to rounding) may need the floor throughout
    assert n_floor <= max(64, max_floor_frac * r.size), f"{label}: too many floor-only passes ({rep})"
    return rep


def check_dw(gpu, ref, name_out: str, scale, label: str = ""):
    """dW / dB: relative L2 <= 1e-4 (FP32 output) or 1 ulp of the rounded
    oracle (16-bit output).  A column sums thousands of rows in FP32 and its
    value is typically ~1/sqrt(M) of the summed magnitudes, so its
    cancellation floor is 2^-16 of those magnitudes for every type and many
    columns may need it; the relative-L2 bar still holds for all of them."""
    rep = check(gpu, ref, name_out, scale=scale, label=label, max_floor_frac=0.5, floor=2.0 ** -16)
    if name_out == "float32":
        assert rep["rel_l2"] <= DW_REL_L2, f"{label}: relative L2 {rep['rel_l2']:.3g} > {DW_REL_L2}"
    return rep
