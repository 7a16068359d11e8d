"""The autograd layer: gradients against the FP64 oracle, frozen
parameters get no gradient (and the same input gradient), and nothing is
computed for a backward when nothing requires grad ("perf(norm): skip dW/dB
calculation when parameters are frozen", Key Changes and Test Validation)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_util import bits_equal, dw_scale, f64, unit_xhat
from tolerance import check, check_dw, rounded

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def A():
    from conftest import built_package
    built_package()
    from row_normalization_rmsnorm_gb300 import autograd
    return autograd


def _case(shape, seed, **kw):
    M = int(np.prod(shape[:-1]))
    c = si.norm_case(M, shape[-1], seed=seed, dtype="bfloat16", **kw)
    return {k: (v.view(*shape) if v.dim() == 2 else v) for k, v in c.items()}


def test_rms_norm_autograd_trainable_and_frozen(A):
    c = _case((4, 96, 1024), 31, gemma=True, with_bias=False)
    x = c["x"].cuda().requires_grad_()
    w = c["w"].cuda().requires_grad_()
    dy = c["dy"].cuda()
    y = A.rms_norm(x, w, EPS, 1.0)
    gx, gw = torch.autograd.grad(y, (x, w), dy)
    x64, dy64, w64 = f64(c["x"].view(-1, 1024)), f64(c["dy"].view(-1, 1024)), f64(c["w"])
    ry, rr = oracle.rms_fwd(x64, w64, 1.0, EPS)
    rdx, rdw, sc = oracle.rms_bwd(x64, dy64, w64, 1.0, EPS, with_scale=True, rstd=rr)
    check(y.view(-1, 1024), ry, "bfloat16", label="autograd rms y")
    check(gx.view(-1, 1024), rdx, "bfloat16", scale=sc, label="autograd rms dx")
    check_dw(gw, rdw, "bfloat16", dw_scale(dy64, unit_xhat(x64, False, EPS)), label="autograd rms dw")
    # frozen weight: no weight gradient, the same input gradient
    wf = c["w"].cuda()
    xf = c["x"].cuda().requires_grad_()
    yf = A.rms_norm(xf, wf, EPS, 1.0)
    yf.backward(dy)
    assert wf.grad is None
    assert bits_equal(xf.grad, gx)


def test_rms_norm_in_place_backward(A):
    # in_place=True: the input gradient is written over the incoming output
    # gradient's storage, with the bits of the out-of-place call and the
    # oracle's values
    c = _case((4, 96, 1024), 35, gemma=True, with_bias=False)
    x = c["x"].cuda().requires_grad_()
    w = c["w"].cuda().requires_grad_()
    dy = c["dy"].cuda()
    gx, gw = torch.autograd.grad(A.rms_norm(x, w, EPS, 1.0), (x, w), dy.clone())
    dy_in = dy.clone()
    gx2, gw2 = torch.autograd.grad(A.rms_norm(x, w, EPS, 1.0, in_place=True), (x, w), dy_in)
    assert bits_equal(gx, gx2) and bits_equal(gw, gw2)
    assert gx2.data_ptr() == dy_in.data_ptr(), "dx was not written over dy"
    assert bits_equal(dy_in, gx2)
    x64, dy64, w64 = f64(c["x"].view(-1, 1024)), f64(c["dy"].view(-1, 1024)), f64(c["w"])
    _, rr = oracle.rms_fwd(x64, w64, 1.0, EPS)
    rdx, _, sc = oracle.rms_bwd(x64, dy64, w64, 1.0, EPS, with_scale=True, rstd=rr)
    check(gx2.view(-1, 1024), rdx, "bfloat16", scale=sc, label="autograd rms in-place dx")
    # the module form
    m = A.RMSNorm(1024, EPS, offset=1.0, in_place=True)
    with torch.no_grad():
        m.weight.copy_(w)
    y = m(x)
    dy_m = dy.clone()
    (gxm,) = torch.autograd.grad(y, (x,), dy_m)
    assert bits_equal(gxm, gx) and gxm.data_ptr() == dy_m.data_ptr()


def test_layer_norm_weight_and_bias_are_independent(A):
    c = _case((512, 2048), 32)
    dy = c["dy"].cuda()
    grads = {}
    for wt, bt in [(True, True), (True, False), (False, True), (False, False)]:
        x = c["x"].cuda().requires_grad_()
        w = c["w"].cuda().requires_grad_(wt)
        b = c["b"].cuda().requires_grad_(bt)
        A.layer_norm(x, w, b, EPS).backward(dy)
        assert (w.grad is not None) == wt and (b.grad is not None) == bt
        grads[(wt, bt)] = (x.grad, w.grad, b.grad)
    ref = grads[(True, True)][0]
    for k, (gx, _, _) in grads.items():
        assert bits_equal(gx, ref), k
    x64, dy64, w64 = f64(c["x"]), f64(c["dy"]), f64(c["w"])
    _, mean, rstd, _ = oracle.ln_fwd(x64, w64, f64(c["b"]), 0.0, EPS)
    rdx, rdw, rdb, sc = oracle.ln_bwd(x64, dy64, w64, 0.0, EPS, with_scale=True, mean=mean, rstd=rstd)
    check(ref, rdx, "bfloat16", scale=sc, label="autograd ln dx")
    check_dw(grads[(True, True)][1], rdw, "bfloat16", dw_scale(dy64, unit_xhat(x64, True, EPS)), label="ln dw")
    check_dw(grads[(True, True)][2], rdb, "bfloat16", np.abs(dy64).sum(0), label="ln db")


def test_fused_add_autograd(A):
    c = _case((2, 64, 4096), 33, with_bias=False, fused_add=True)
    x = c["x"].cuda().requires_grad_()
    r = c["residual"].cuda().requires_grad_()
    w = c["w"].cuda().requires_grad_()
    y, h = A.fused_add_rms_norm(x, r, w, EPS)
    gx, gr, gw = torch.autograd.grad((y, h), (x, r, w), (c["dy"].cuda(), c["dh_out"].cuda()))
    assert bits_equal(gx, gr)
    N = 4096
    x64, r64, dy64, dh64, w64 = (f64(c[k].reshape(-1, N)) if c[k].dim() > 1 else f64(c[k])
                                 for k in ("x", "residual", "dy", "dh_out", "w"))
    ry, rh, rr = oracle.fused_add_rms_fwd(x64, r64, w64, 0.0, EPS)
    hs = rounded(rh, "bfloat16")
    rdx, rdw, sc = oracle.fused_add_rms_bwd(hs, dy64, w64, dh64, 0.0, EPS, with_scale=True, rstd=rr)
    check(y.reshape(-1, N), ry, "bfloat16", label="autograd fadd y")
    check(gx.reshape(-1, N), rdx, "bfloat16", scale=sc, label="autograd fadd dx")
    check_dw(gw, rdw, "bfloat16", dw_scale(dy64, unit_xhat(hs, False, EPS)), label="autograd fadd dw")


def test_fused_add_in_place_backward(A):
    # in_place=True: dx is written over the residual stream's incoming
    # gradient, with the bits of the out-of-place call
    c = _case((2, 64, 4096), 36, with_bias=False, fused_add=True)
    x = c["x"].cuda().requires_grad_()
    r = c["residual"].cuda().requires_grad_()
    w = c["w"].cuda().requires_grad_()
    dy, dh = c["dy"].cuda(), c["dh_out"].cuda()
    ref = torch.autograd.grad(A.fused_add_rms_norm(x, r, w, EPS, 1.0), (x, r, w), (dy.clone(), dh.clone()))
    dh_in = dh.clone()
    out = torch.autograd.grad(A.fused_add_rms_norm(x, r, w, EPS, 1.0, in_place=True), (x, r, w), (dy.clone(), dh_in))
    assert all(bits_equal(a, b) for a, b in zip(ref, out))
    assert out[0].data_ptr() == dh_in.data_ptr(), "dx was not written over dh_out"


def test_no_grad_runs_forward_only(A):
    c = _case((128, 4096), 34, with_bias=False)
    x, w = c["x"].cuda(), c["w"].cuda()
    y = A.rms_norm(x, w)
    assert y.grad_fn is None
    with torch.no_grad():
        y2 = A.rms_norm(x.requires_grad_(), w)
    assert y2.grad_fn is None and bits_equal(y, y2)


def test_modules(A):
    torch.manual_seed(0)
    m = A.RMSNorm(4096, offset=1.0)
    ln = A.LayerNorm(4096)
    fa = A.FusedAddRMSNorm(4096)
    x = torch.randn(3, 7, 4096, device="cuda").to(torch.bfloat16)
    r = torch.randn(3, 7, 4096, device="cuda").to(torch.bfloat16)
    y = m(x)
    # zero weight with offset 1: plain RMS normalisation
    ref = oracle.rms_fwd(f64(x.view(-1, 4096).cpu()), np.zeros(4096), 1.0, 1e-6)[0]
    check(y.view(-1, 4096), ref, "bfloat16", label="module rms")
    (ln(x).float().sum() + fa(x, r)[0].float().sum()).backward()
    assert ln.weight.grad is not None and ln.bias.grad is not None and fa.weight.grad is not None
