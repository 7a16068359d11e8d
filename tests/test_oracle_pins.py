"""Pins of the FP64 oracle against things other than itself (CPU only).

Each oracle function is checked against at least one of: a library special
case (torch's float64 CPU rms_norm / layer_norm with autograd), central finite
differences of its own pinned forward, closed forms, per-row invariants, the
worked BF16 example printed on "fix(cutedsl): fuse Gemma RMSNorm weight offset
in FP32" (Summary) and a brute-force check of the rounding helpers over every
16-bit pattern.  A dropped term, a wrong sign, a transposed operand or eps in
the wrong place fails at least one test here.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synthetic_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            out[k] = float(v)
    return out


def rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# Rounding helpers
# --------------------------------------------------------------------------

def _all_patterns(torch_dtype):
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch_dtype).double().numpy()
    pats = np.arange(0, 1 << 16, dtype=np.uint16)
    return pats, vals


@pytest.mark.parametrize("dtype,tdt", [("bfloat16", torch.bfloat16),
                                       ("float16", torch.float16)])
def test_round_every_pattern_is_fixed_point(dtype, tdt):
    pats, vals = _all_patterns(tdt)
    ok = ~np.isnan(vals)
    got = oracle.round_to(vals[ok], dtype)
    assert np.array_equal(got, pats[ok])


@pytest.mark.parametrize("dtype,tdt", [("bfloat16", torch.bfloat16),
                                       ("float16", torch.float16)])
def test_round_midpoints_tie_to_even(dtype, tdt):
    pats, vals = _all_patterns(tdt)
    # positive finite values in increasing order: patterns 0x0000 .. max finite
    pos = vals[: (0x7F80 if dtype == "bfloat16" else 0x7C00)]
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2.0                       # exact in FP64
    lo_bits = np.arange(0, len(lo), dtype=np.uint16)
    hi_bits = lo_bits + 1
    even = np.where(lo_bits % 2 == 0, lo_bits, hi_bits)
    assert np.array_equal(oracle.round_to(mid, dtype), even)
    up = np.nextafter(mid, np.inf)
    dn = np.nextafter(mid, -np.inf)
    assert np.array_equal(oracle.round_to(up, dtype), hi_bits)
    assert np.array_equal(oracle.round_to(dn, dtype), lo_bits)
    # the same with the sign bit set
    assert np.array_equal(oracle.round_to(-up, dtype), hi_bits | 0x8000)


def test_round_overflow_and_specials():
    # bf16: max finite (2 - 2^-7) * 2^127; halfway to 2^128 ties to "even" 2^128 -> inf
    maxb = (2 - 2 ** -7) * 2.0 ** 127
    half = 2.0 ** (127 - 8)
    assert oracle.round_bf16_bits(maxb) == 0x7F7F
    assert oracle.round_bf16_bits(maxb + half) == 0x7F80
    assert oracle.round_bf16_bits(np.nextafter(maxb + half, 0)) == 0x7F7F
    assert oracle.round_bf16_bits(-math.inf) == 0xFF80
    assert oracle.round_f16_bits(65504.0) == 0x7BFF
    assert oracle.round_f16_bits(65520.0) == 0x7C00
    assert oracle.round_f16_bits(np.nextafter(65520.0, 0)) == 0x7BFF
    assert oracle.round_f16_bits(2.0 ** -25) == 0x0000      # tie to even (0)
    assert oracle.round_f16_bits(np.nextafter(2.0 ** -25, 1)) == 0x0001
    assert oracle.round_f16_bits(-0.0) == 0x8000
    assert oracle.round_bf16_bits(float("nan")) & 0x7F80 == 0x7F80


def test_round_bf16_matches_torch_on_fp32_values():
    # torch converts float32 -> bfloat16 with round-to-nearest-even; on values
    # exactly representable in float32 the direct FP64 rounding must agree.
    r = rng(1)
    v = (r.standard_normal(200000) * np.exp2(r.integers(-130, 120, 200000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_to(v.astype(np.float64), "bfloat16")
    assert np.array_equal(got, ref)


def test_round_f16_matches_numpy_on_doubles():
    # numpy converts float64 -> float16 directly (no float32 step), RNE.
    r = rng(2)
    v = r.standard_normal(200000) * np.exp2(r.integers(-28, 17, 200000))
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    got = oracle.round_to(v, "float16")
    assert np.array_equal(got, ref)


def test_round_f32_matches_numpy():
    v = rng(3).standard_normal(10000) * 1e3
    assert np.array_equal(oracle.round_to(v, "float32"), v.astype(np.float32))


def test_round_is_direct_not_double_rounded():
    # A value just above a bf16 midpoint, but which FP32 would round down onto
    # the midpoint, must still round up when rounded directly from FP64.
    mid = 1.0 + 2.0 ** -8          # halfway between 1.0 and 1.0078125
    v = mid + 2.0 ** -30           # rounds to mid in float32
    assert float(np.float32(v)) == mid
    assert oracle.round_bf16_bits(v) == 0x3F81   # 1.0078125


# --------------------------------------------------------------------------
# The worked example of the Gemma offset (golden, from the pages)
# --------------------------------------------------------------------------

def test_worked_example_bf16_preadd_vs_fp32_sum():
    g = read_golden_kv("gemma_offset_worked_example.txt")
    w, off = g["weight"], g["offset"]
    assert oracle.round_bf16_bits(w) == 0x3B80                 # 2^-8 is exact in bf16
    pre = torch.tensor([oracle.round_bf16_bits(w + off)], dtype=torch.int32)
    pre = pre.to(torch.int16).view(torch.bfloat16).double().item()
    assert pre == g["bf16_preadded"]
    assert float(np.float32(w) + np.float32(off)) == g["fp32_sum"]


def test_worked_example_in_oracle_forward():
    g = read_golden_kv("gemma_offset_worked_example.txt")
    N = 8
    w = np.full(N, g["weight"])
    # x constant 1, eps 0: rstd = 1 and y_j = w_j + offset exactly
    y, rstd = oracle.rms_fwd(np.ones((1, N)), w, offset=g["offset"], eps=0.0)
    assert rstd[0] == 1.0
    assert np.all(y == g["fp32_sum"])
    # negative control: the BF16 pre-added weight loses the offset's low bits
    y_pre, _ = oracle.rms_fwd(np.ones((1, N)), np.full(N, g["bf16_preadded"]),
                              offset=0.0, eps=0.0)
    assert np.all(y_pre == 1.0)
    # a BF16 output at xhat = 1.5: 1.5 * 1.00390625 rounds to 1.5078125, the
    # pre-added weight gives 1.5
    # (row [1.5]*3 + [0.5]*5 has mean square exactly 1, so xhat = x)
    x15 = np.array([[1.5] * 3 + [0.5] * 5])
    y15, r15 = oracle.rms_fwd(x15, w, offset=g["offset"], eps=0.0)
    assert r15[0] == 1.0 and y15[0, 0] == 1.5 * g["fp32_sum"]
    bits = oracle.round_to(y15[0, :3], "bfloat16")
    assert np.all(bits == 0x3FC1)      # 1.5078125
    y15p, _ = oracle.rms_fwd(x15, np.full(N, 1.0), offset=0.0, eps=0.0)
    assert np.all(oracle.round_to(y15p[0, :3], "bfloat16") == 0x3FC0)   # 1.5


def test_preadd_control_reaches_the_pages_before_magnitude():
    """Pre-adding the offset in BF16 moves Y by the order of the pages'
    "before" error (~3e-3 relative L2); the FP32-fused offset does not."""
    table = {}
    with open(os.path.join(GOLDEN, "gemma_repro_error_magnitudes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                op, out, before, after = line.split()
                table[(op, out)] = (float(before), float(after))
    case = si.norm_case(128, 4096, seed=42, dtype="bfloat16", gemma=True,
                        with_bias=False)
    x = case["x"].double().numpy()
    w = case["w"].double().numpy()
    w_pre = torch.from_numpy(oracle.round_to(w + 1.0, "bfloat16").view(np.int16)) \
        .view(torch.bfloat16).double().numpy()
    y, _ = oracle.rms_fwd(x, w, offset=1.0, eps=1e-6)
    y_pre, _ = oracle.rms_fwd(x, w_pre, offset=0.0, eps=1e-6)
    rel = np.linalg.norm(y_pre - y) / np.linalg.norm(y)
    before = table[("RMSNorm", "Y")][0]
    assert before / 3 < rel < before * 3, rel
    # output rounding alone (what a correct BF16 kernel adds) stays well below
    y_b = torch.from_numpy(oracle.round_to(y, "bfloat16").view(np.int16)) \
        .view(torch.bfloat16).double().numpy()
    assert np.linalg.norm(y_b - y) / np.linalg.norm(y) < before


# --------------------------------------------------------------------------
# Library special cases: torch float64 CPU ops + autograd
# --------------------------------------------------------------------------

SHAPES = [(1, 1), (3, 7), (5, 64), (4, 513)]


def _t(a, grad=False):
    return torch.tensor(a, dtype=torch.float64, requires_grad=grad)


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("offset,eps", [(0.0, 1e-6), (1.0, 1e-6), (0.5, 0.3)])
def test_rms_matches_torch_float64(M, N, offset, eps):
    r = rng(M * 100 + N)
    x = r.standard_normal((M, N))
    w = 0.1 * r.standard_normal(N) + (0.0 if offset else 1.0)
    dy = r.standard_normal((M, N))
    y, rstd = oracle.rms_fwd(x, w, offset, eps)
    dx, dw, _ = oracle.rms_bwd(x, dy, w, offset, eps)
    xt, wt = _t(x, True), _t(w, True)
    yt = F.rms_norm(xt, (N,), wt + offset, eps)
    gx, gw = torch.autograd.grad(yt, (xt, wt), _t(dy))
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dx, gx.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dw, gw.numpy(), rtol=1e-10, atol=1e-11)
    ms = (x * x).mean(axis=1)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(ms + eps), rtol=1e-13)
    # the saved-statistic path is the same computation
    dxs, dws, _ = oracle.rms_bwd(x, dy, w, offset, eps, rstd=rstd)
    np.testing.assert_array_equal(dxs, dx)
    np.testing.assert_array_equal(dws, dw)


def test_saved_statistics_enter_the_formula():
    # a perturbed saved rstd moves dx as the formula says: with rstd' = s*rstd
    # every term is rescaled, dx' = s*rstd*(g - s*xhat*s*c)
    r = rng(77)
    x, dy = r.standard_normal((3, 40)), r.standard_normal((3, 40))
    w = 1 + 0.1 * r.standard_normal(40)
    _, rstd = oracle.rms_fwd(x, w, 0.0, 1e-6)
    s = 1.001
    dx2, _, _ = oracle.rms_bwd(x, dy, w, 0.0, 1e-6, rstd=rstd * s)
    rs = (rstd * s)[:, None]
    xh = x * rs
    g = dy * w
    c = (g * xh).mean(axis=1, keepdims=True)
    np.testing.assert_allclose(dx2, rs * (g - xh * c), rtol=1e-12, atol=1e-14)
    _, mean, rstd_l, _ = oracle.ln_fwd(x, w, None, 0.0, 1e-6)
    dxl, _, _, _ = oracle.ln_bwd(x, dy, w, 0.0, 1e-6, mean=mean + 0.01, rstd=rstd_l)
    xh = (x - (mean + 0.01)[:, None]) * rstd_l[:, None]
    expect = rstd_l[:, None] * (g - g.mean(1, keepdims=True) - xh * (g * xh).mean(1, keepdims=True))
    np.testing.assert_allclose(dxl, expect, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("M,N", SHAPES[1:])
@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("offset,eps", [(0.0, 1e-6), (1.0, 1e-5)])
def test_ln_matches_torch_float64(M, N, with_bias, offset, eps):
    r = rng(M * 1000 + N + with_bias)
    x = r.standard_normal((M, N)) * 2 + 0.5
    w = 1 + 0.1 * r.standard_normal(N)
    b = 0.1 * r.standard_normal(N) if with_bias else None
    dy = r.standard_normal((M, N))
    y, mean, rstd, _ = oracle.ln_fwd(x, w, b, offset, eps)
    dx, dw, db, _ = oracle.ln_bwd(x, dy, w, offset, eps)
    xt, wt = _t(x, True), _t(w, True)
    bt = _t(b, True) if with_bias else _t(np.zeros(N), True)
    yt = F.layer_norm(xt, (N,), wt + offset, bt, eps)
    gx, gw, gb = torch.autograd.grad(yt, (xt, wt, bt), _t(dy))
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dx, gx.numpy(), rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(dw, gw.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(db, gb.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(x.var(axis=1) + eps), rtol=1e-12)
    dxs, dws, dbs, _ = oracle.ln_bwd(x, dy, w, offset, eps, mean=mean, rstd=rstd)
    np.testing.assert_array_equal(dxs, dx)
    np.testing.assert_array_equal(dws, dw)
    np.testing.assert_array_equal(dbs, db)


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_fused_add_matches_torch_float64(M, N, offset):
    r = rng(M * 7 + N)
    x = r.standard_normal((M, N))
    res = r.standard_normal((M, N))
    w = 0.1 * r.standard_normal(N) + (0.0 if offset else 1.0)
    dy = r.standard_normal((M, N))
    dho = r.standard_normal((M, N))
    eps = 1e-6
    y, h, rstd = oracle.fused_add_rms_fwd(x, res, w, offset, eps)
    xt, rt, wt = _t(x, True), _t(res, True), _t(w, True)
    ht = xt + rt
    yt = F.rms_norm(ht, (N,), wt + offset, eps)
    gx, gr, gw = torch.autograd.grad((yt, ht), (xt, rt, wt), (_t(dy), _t(dho)))
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(h, x + res)
    # backward at the (here unrounded) saved h
    dx, dw, _ = oracle.fused_add_rms_bwd(h, dy, w, dho, offset, eps)
    np.testing.assert_allclose(dx, gx.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dx, gr.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dw, gw.numpy(), rtol=1e-10, atol=1e-11)
    # the forward's saved rstd gives the same result at the unrounded h
    dxs, dws, _ = oracle.fused_add_rms_bwd(h, dy, w, dho, offset, eps, rstd=rstd)
    np.testing.assert_array_equal(dxs, dx)
    np.testing.assert_array_equal(dws, dw)
    # without a residual-output gradient it reduces to the RMSNorm backward
    dx0, dw0, _ = oracle.fused_add_rms_bwd(h, dy, w, None, offset, eps)
    dxr, dwr, _ = oracle.rms_bwd(h, dy, w, offset, eps)
    np.testing.assert_array_equal(dx0, dxr)
    np.testing.assert_array_equal(dw0, dwr)


# --------------------------------------------------------------------------
# Central finite differences of the (pinned) forwards
# --------------------------------------------------------------------------

def _fd(f, a, h=1e-6):
    g = np.zeros_like(a)
    it = np.nditer(a, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        ap = a.copy(); ap[idx] += h
        am = a.copy(); am[idx] -= h
        g[idx] = (f(ap) - f(am)) / (2 * h)
    return g


@pytest.mark.parametrize("M,N", [(2, 4), (3, 9), (2, 16)])
def test_rms_bwd_finite_differences(M, N):
    r = rng(10 + N)
    x, dy = r.standard_normal((M, N)), r.standard_normal((M, N))
    w, off, eps = r.standard_normal(N) * 0.3, 1.0, 1e-3
    loss = lambda xx, ww: float((oracle.rms_fwd(xx, ww, off, eps)[0] * dy).sum())
    dx, dw, _ = oracle.rms_bwd(x, dy, w, off, eps)
    np.testing.assert_allclose(dx, _fd(lambda a: loss(a, w), x), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dw, _fd(lambda a: loss(x, a), w), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("M,N", [(2, 4), (3, 9), (2, 16)])
def test_ln_bwd_finite_differences(M, N):
    r = rng(20 + N)
    x, dy = r.standard_normal((M, N)), r.standard_normal((M, N))
    w, b, off, eps = 1 + 0.2 * r.standard_normal(N), r.standard_normal(N), 0.25, 1e-3
    loss = lambda xx, ww, bb: float((oracle.ln_fwd(xx, ww, bb, off, eps)[0] * dy).sum())
    dx, dw, db, _ = oracle.ln_bwd(x, dy, w, off, eps)
    np.testing.assert_allclose(dx, _fd(lambda a: loss(a, w, b), x), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dw, _fd(lambda a: loss(x, a, b), w), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(db, _fd(lambda a: loss(x, w, a), b), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("M,N", [(2, 4), (3, 11)])
def test_fused_add_bwd_finite_differences(M, N):
    r = rng(30 + N)
    x, res = r.standard_normal((M, N)), r.standard_normal((M, N))
    dy, dho = r.standard_normal((M, N)), r.standard_normal((M, N))
    w, off, eps = 0.1 * r.standard_normal(N), 1.0, 1e-3

    def loss(xx, rr, ww):
        y, h, _ = oracle.fused_add_rms_fwd(xx, rr, ww, off, eps)
        return float((y * dy).sum() + (h * dho).sum())

    h = x + res
    dx, dw, _ = oracle.fused_add_rms_bwd(h, dy, w, dho, off, eps)
    np.testing.assert_allclose(dx, _fd(lambda a: loss(a, res, w), x), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dx, _fd(lambda a: loss(x, a, w), res), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(dw, _fd(lambda a: loss(x, res, a), w), rtol=1e-6, atol=1e-7)


# --------------------------------------------------------------------------
# Per-row invariants and closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_rms_scale_invariance_closed_form(eps):
    # sum_j x_j dx_j = rstd * sum_j g_j x_j * eps / (mean(x^2) + eps)
    r = rng(40)
    M, N = 6, 257
    x, dy = r.standard_normal((M, N)) * 1.7, r.standard_normal((M, N))
    w, off = 0.1 * r.standard_normal(N), 1.0
    dx, _, _ = oracle.rms_bwd(x, dy, w, off, eps)
    ms = (x * x).mean(axis=1)
    rs = 1 / np.sqrt(ms + eps)
    g = dy * (w + off)
    expect = rs * (g * x).sum(axis=1) * eps / (ms + eps)
    np.testing.assert_allclose((x * dx).sum(axis=1), expect, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_ln_invariants(eps):
    r = rng(41)
    M, N = 6, 300
    x, dy = r.standard_normal((M, N)) * 3 + 2, r.standard_normal((M, N))
    w = 1 + 0.1 * r.standard_normal(N)
    dx, _, _, _ = oracle.ln_bwd(x, dy, w, 0.0, eps)
    # sum_j dx_j = 0
    np.testing.assert_allclose(dx.sum(axis=1), 0.0, atol=1e-12)
    # sum_j xhat_j dx_j = rstd * sum_j g_j xhat_j * eps / (var + eps)
    mu, var = x.mean(axis=1, keepdims=True), x.var(axis=1, keepdims=True)
    rs = 1 / np.sqrt(var + eps)
    xh = (x - mu) * rs
    g = dy * w
    expect = (rs * (g * xh).sum(axis=1, keepdims=True) * eps / (var + eps)).ravel()
    np.testing.assert_allclose((xh * dx).sum(axis=1), expect, rtol=1e-8, atol=1e-12)


def test_closed_forms_constant_rows_and_single_row():
    N, c, eps = 10, 0.75, 1e-2
    x = np.full((1, N), c)
    w = np.linspace(0.5, 1.5, N)
    y, rstd = oracle.rms_fwd(x, w, 0.0, eps)
    np.testing.assert_allclose(y[0], c / math.sqrt(c * c + eps) * w, rtol=1e-15)
    b = np.linspace(-1, 1, N)
    yl, mean, rs, _ = oracle.ln_fwd(x, w, b, 0.0, eps)
    np.testing.assert_allclose(yl[0], b, atol=1e-15)          # xhat = 0 -> y = b
    assert mean[0] == c and rs[0] == pytest.approx(1 / math.sqrt(eps))
    # M = 1: dW = dy * xhat and dB = dy exactly
    r = rng(42)
    x1, dy1 = r.standard_normal((1, N)), r.standard_normal((1, N))
    _, dw, _ = oracle.rms_bwd(x1, dy1, w, 0.0, eps)
    rr = 1 / math.sqrt((x1 * x1).mean() + eps)
    np.testing.assert_allclose(dw, dy1[0] * x1[0] * rr, rtol=1e-14)
    _, dwl, dbl, _ = oracle.ln_bwd(x1, dy1, w, 0.0, eps)
    xh = (x1[0] - x1.mean()) / math.sqrt(x1.var() + eps)
    np.testing.assert_allclose(dwl, dy1[0] * xh, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(dbl, dy1[0])


def test_frozen_outputs_do_not_change_dx():
    r = rng(43)
    x, dy = r.standard_normal((5, 33)), r.standard_normal((5, 33))
    w = 1 + 0.1 * r.standard_normal(33)
    a = oracle.rms_bwd(x, dy, w, 0.0, 1e-6, compute_dw=True)[0]
    b = oracle.rms_bwd(x, dy, w, 0.0, 1e-6, compute_dw=False)[0]
    np.testing.assert_array_equal(a, b)
    a = oracle.ln_bwd(x, dy, w, 0.0, 1e-6, True, True)[0]
    b = oracle.ln_bwd(x, dy, w, 0.0, 1e-6, False, False)[0]
    np.testing.assert_array_equal(a, b)


def test_scale_outputs_bound_the_result():
    # the *_scale diagnostics are magnitudes of the summed terms: |out| <= scale
    r = rng(44)
    x, dy = r.standard_normal((4, 50)), r.standard_normal((4, 50))
    w, b = 1 + 0.1 * r.standard_normal(50), r.standard_normal(50)
    dx, _, sc = oracle.rms_bwd(x, dy, w, 1.0, 1e-6, with_scale=True)
    assert np.all(np.abs(dx) <= sc * (1 + 1e-12))
    dx, _, _, sc = oracle.ln_bwd(x, dy, w, 0.0, 1e-6, with_scale=True)
    assert np.all(np.abs(dx) <= sc * (1 + 1e-12))
    y, _, _, sc = oracle.ln_fwd(x, w, b, 0.0, 1e-6, with_scale=True)
    assert np.all(np.abs(y) <= sc * (1 + 1e-12))
