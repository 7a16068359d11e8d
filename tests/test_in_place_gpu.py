"""In-place backward against the FP64 oracle.

"fix(cutedsl): fuse Gemma RMSNorm weight offset in FP32" (Testing Done,
supplemental diagnostics) covers in-place as well as out-of-place backward.
Here the input gradient is written over its own upstream gradient: dx == dy
for RMSNorm and LayerNorm, dx == dh_out for FusedAddRMSNorm (whose gradient
serves both x and the residual).  Each layout -- contiguous rows, row stride
N + 64 (16-byte aligned rows: the staged kernels) and a base one element off
16-byte alignment (the general kernels) -- is compared element by element
with the oracle, dW / dB included, and the padding between strided rows must
keep its NaN sentinels.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_util import Strided, dw_scale, f64, unit_xhat, workspace
from tolerance import check, check_dw, dtype_name, rounded

pytestmark = pytest.mark.gpu

EPS = 1e-6
LAYOUTS = [("contiguous", None, 0), ("stride+64", 64, 0), ("misaligned", 64, 1)]


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def layout(N, extra, lead):
    return (None if extra is None else N + extra), lead


@pytest.mark.parametrize("name,extra,lead", LAYOUTS)
@pytest.mark.parametrize("M,N", [(300, 4096), (67, 1024)])
def test_rms_backward_in_place(g, name, extra, lead, M, N):
    case = si.norm_case(M, N, seed=21, dtype="bfloat16", with_bias=False)
    stride, lead = layout(N, extra, lead)
    X = Strided.of(case["x"], stride, lead)
    DY = Strided.of(case["dy"], stride, lead)   # becomes dx
    Y = Strided(M, N, torch.bfloat16, stride, lead)
    w = case["w"].cuda()
    rstd = torch.empty(M, device="cuda")
    dw = torch.empty(N, dtype=torch.float32, device="cuda")
    g.norm_rms_fwd(X.view, w, Y.view, rstd, 1.0, EPS)
    g.norm_rms_bwd(DY.view, X.view, w, rstd, DY.view, dw, workspace(g, M, N, True), 1.0, EPS)
    torch.cuda.synchronize()
    x, dy, w64 = f64(case["x"]), f64(case["dy"]), f64(case["w"])
    _, r = oracle.rms_fwd(x, w64, 1.0, EPS)
    dx, dwr, sc = oracle.rms_bwd(x, dy, w64, 1.0, EPS, with_scale=True, rstd=r)
    check(DY.view, dx, "bfloat16", scale=sc, label=f"in-place rms {name} {M}x{N} dx")
    check_dw(dw, dwr, "float32", dw_scale(dy, unit_xhat(x, False, EPS)), label=f"in-place rms {name} dw")
    assert DY.padding_intact() and X.padding_intact()


@pytest.mark.parametrize("name,extra,lead", LAYOUTS)
def test_ln_backward_in_place(g, name, extra, lead):
    M, N = 300, 4096
    case = si.norm_case(M, N, seed=22, dtype="bfloat16")
    stride, lead = layout(N, extra, lead)
    X = Strided.of(case["x"], stride, lead)
    DY = Strided.of(case["dy"], stride, lead)
    Y = Strided(M, N, torch.bfloat16, stride, lead)
    w, b = case["w"].cuda(), case["b"].cuda()
    mean, rstd = torch.empty(M, device="cuda"), torch.empty(M, device="cuda")
    dw = torch.empty(N, dtype=torch.float32, device="cuda")
    db = torch.empty(N, dtype=torch.float32, device="cuda")
    g.norm_ln_fwd(X.view, w, b, Y.view, mean, rstd, 0.0, EPS)
    g.norm_ln_bwd(DY.view, X.view, w, mean, rstd, DY.view, dw, db, workspace(g, M, N, True, True), 0.0, EPS)
    torch.cuda.synchronize()
    x, dy, w64 = f64(case["x"]), f64(case["dy"]), f64(case["w"])
    _, mu, r, _ = oracle.ln_fwd(x, w64, f64(case["b"]), 0.0, EPS)
    dx, dwr, dbr, sc = oracle.ln_bwd(x, dy, w64, 0.0, EPS, with_scale=True, mean=mu, rstd=r)
    check(DY.view, dx, "bfloat16", scale=sc, label=f"in-place ln {name} dx")
    check_dw(dw, dwr, "float32", dw_scale(dy, unit_xhat(x, True, EPS)), label=f"in-place ln {name} dw")
    check_dw(db, dbr, "float32", np.abs(dy).sum(0), label=f"in-place ln {name} db")
    assert DY.padding_intact() and X.padding_intact()


@pytest.mark.parametrize("name,extra,lead", LAYOUTS)
@pytest.mark.parametrize("trainable", [True, False])
def test_fused_add_backward_in_place(g, name, extra, lead, trainable):
    M, N = 300, 4096
    case = si.norm_case(M, N, seed=23, dtype="bfloat16", gemma=True, with_bias=False, fused_add=True)
    stride, lead = layout(N, extra, lead)
    X = Strided.of(case["x"], stride, lead)
    R = Strided.of(case["residual"], stride, lead)
    DY = Strided.of(case["dy"], stride, lead)
    DH = Strided.of(case["dh_out"], stride, lead)   # becomes dx (= d residual)
    Y, H = (Strided(M, N, torch.bfloat16, stride, lead) for _ in range(2))
    w = case["w"].cuda()
    rstd = torch.empty(M, device="cuda")
    dw = torch.empty(N, dtype=torch.float32, device="cuda") if trainable else None
    g.norm_fused_add_rms_fwd(X.view, R.view, w, Y.view, H.view, rstd, 1.0, EPS)
    g.norm_fused_add_rms_bwd(DY.view, DH.view, H.view, w, rstd, DH.view, dw,
                             workspace(g, M, N, trainable), 1.0, EPS)
    torch.cuda.synchronize()
    x, r, dy, dh, w64 = (f64(case[k]) for k in ("x", "residual", "dy", "dh_out", "w"))
    _, h, rs = oracle.fused_add_rms_fwd(x, r, w64, 1.0, EPS)
    h16 = rounded(h, "bfloat16")   # the backward works at the saved, rounded h
    dx, dwr, sc = oracle.fused_add_rms_bwd(h16, dy, w64, dh, 1.0, EPS, with_scale=True, rstd=rs)
    check(DH.view, dx, "bfloat16", scale=sc, label=f"in-place fadd {name} dx")
    if trainable:
        check_dw(dw, dwr, "float32", dw_scale(dy, unit_xhat(h16, False, EPS)), label=f"in-place fadd {name} dw")
    assert DH.padding_intact() and H.padding_intact()
