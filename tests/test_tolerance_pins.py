"""Pins of the parity machinery itself (CPU only).

The GPU parity checks accept an element when it is within one ulp of the
rounded oracle (16-bit outputs) or within 1e-5 relative (FP32), or, for
outputs formed by cancellation, within floor * scale, where scale is the
oracle's magnitude of the terms summed into that element.  These tests make
sure that machinery can fail:

* check() rejects a 2-ulp BF16 error, a 2e-5 relative FP32 error whose scale
  equals the value, and floor-only passes just above the 1 % cap;
* check_dw() rejects an FP32 dW off by 2e-4 relative L2;
* the oracle's *_scale outputs equal hand-computed values on 1 x 4 rows, so
  a scale that is too large (which would widen the floor clause) fails here.
"""
import numpy as np
import pytest
import torch

import oracle
from tolerance import FLOOR, check, check_dw, rounded, ulp


def bf16_tensor(v64):
    """A BF16 torch tensor holding the given (already representable) values."""
    return torch.from_numpy(np.asarray(v64, np.float64)).to(torch.bfloat16)


def ref_values(n=4096, seed=5):
    r = np.random.default_rng(seed)
    return r.standard_normal(n) * np.exp2(r.integers(-6, 6, n))


def test_exact_rounding_passes_and_two_ulp_fails():
    ref = ref_values()
    good = rounded(ref, "bfloat16")
    rep = check(bf16_tensor(good), ref, "bfloat16", label="exact")
    assert rep["n_floor_only"] == 0
    for scale in (None, np.abs(ref)):
        bad = good.copy()
        bad[17] = good[17] + 2 * ulp(good[17:18], "bfloat16")[0]
        with pytest.raises(AssertionError):
            check(bf16_tensor(bad), ref, "bfloat16", scale=scale, label="2 ulp")


def test_one_ulp_passes():
    ref = ref_values()
    good = rounded(ref, "bfloat16")
    one = good.copy()
    one[3] = good[3] + ulp(good[3:4], "bfloat16")[0]
    check(bf16_tensor(one), ref, "bfloat16", label="1 ulp")


def test_fp32_relative_error_above_the_bar_fails():
    ref = ref_values().astype(np.float32).astype(np.float64)
    g = ref.copy()
    g[9] = ref[9] * (1 + 2e-5)
    # with the scale equal to |value| the floor (2^-17 |value|) cannot rescue it
    with pytest.raises(AssertionError):
        check(torch.from_numpy(g.astype(np.float32)), ref, "float32", scale=np.abs(ref), label="2e-5")
    g[9] = ref[9] * (1 + 5e-6)
    check(torch.from_numpy(g.astype(np.float32)), ref, "float32", scale=np.abs(ref), label="5e-6")


@pytest.mark.parametrize("n_floor,ok", [(100, True), (101, False)])
def test_floor_only_passes_are_capped_at_one_percent(n_floor, ok):
    n = 10000   # cap = max(64, 1 % of n) = 100 elements
    ref = ref_values(n, seed=8)
    good = rounded(ref, "bfloat16")
    scale = np.abs(ref).copy()
    g = good.copy()
    idx = np.arange(n_floor) * 7
    # 1.5 ulp off the rounded value: outside the ulp clause, inside the floor
    # clause because those elements carry a scale 1000 x their value
    g[idx] = good[idx] + 1.5 * ulp(good[idx], "bfloat16")
    scale[idx] = 1000.0 * np.abs(ref[idx])
    assert np.all(1.5 * ulp(good[idx], "bfloat16") <= FLOOR["bfloat16"] * scale[idx] * 1.01)
    gt = torch.from_numpy(g).to(torch.float32)   # 1.5 ulp is not on the BF16 grid; keep it in FP32
    if ok:
        rep = check(gt, ref, "bfloat16", scale=scale, label="cap")
        assert rep["n_floor_only"] == n_floor
    else:
        with pytest.raises(AssertionError, match="too many floor-only"):
            check(gt, ref, "bfloat16", scale=scale, label="cap")


def test_check_dw_rejects_a_relative_l2_error_of_2e_4():
    r = np.random.default_rng(3)
    x, dy = r.standard_normal((64, 256)), r.standard_normal((64, 256))
    w = 1 + 0.1 * r.standard_normal(256)
    _, dw, _ = oracle.rms_bwd(x, dy, w, 0.0, 1e-6)
    xh = oracle.rms_fwd(x, np.ones(256), 0.0, 1e-6)[0]
    scale = np.abs(dy * xh).sum(0)
    check_dw(torch.from_numpy(dw.astype(np.float32)), dw, "float32", scale, label="dw exact")
    with pytest.raises(AssertionError):
        check_dw(torch.from_numpy((dw * (1 + 2e-4)).astype(np.float32)), dw, "float32", scale, label="dw 2e-4")


# ---------------------------------------------------------------------------
# *_scale closed forms on 1 x 4 rows (eps = 0, hand-computed)
# ---------------------------------------------------------------------------
def test_rms_dx_scale_closed_form():
    # x = [1, -1, 1, -1]: mean(x^2) = 1, rstd = 1, xhat = x; w = 1; dy = g = [1, 2, 3, 4]
    # c = sum(g xhat)/N = -2/4; sum |g xhat| / N = 10/4
    # dx = g - xhat c = [1.5, 1.5, 3.5, 3.5]; dx_scale = |g| + |xhat| 2.5
    x = np.array([[1.0, -1.0, 1.0, -1.0]])
    dy = np.array([[1.0, 2.0, 3.0, 4.0]])
    dx, dw, sc = oracle.rms_bwd(x, dy, np.ones(4), 0.0, 0.0, with_scale=True)
    np.testing.assert_array_equal(dx, [[1.5, 1.5, 3.5, 3.5]])
    np.testing.assert_array_equal(sc, [[3.5, 4.5, 5.5, 6.5]])
    np.testing.assert_array_equal(dw, [1.0, -2.0, 3.0, -4.0])
    # the fused-add form adds |dh_out|
    dh = np.array([[0.5, -1.0, 0.0, 2.0]])
    dx, _, sc = oracle.fused_add_rms_bwd(x, dy, np.ones(4), dh, 0.0, 0.0, with_scale=True)
    np.testing.assert_array_equal(dx, [[2.0, 0.5, 3.5, 5.5]])
    np.testing.assert_array_equal(sc, [[4.0, 5.5, 5.5, 8.5]])


def test_ln_scales_closed_form():
    # x = [0, 2, 0, 2]: mean 1, variance 1, rstd 1 (eps = 0), xhat = [-1, 1, -1, 1]
    x = np.array([[0.0, 2.0, 0.0, 2.0]])
    w = np.array([1.0, 2.0, 1.0, 2.0])
    b = np.array([0.5, 0.0, -0.5, 0.0])
    y, mean, rstd, ysc = oracle.ln_fwd(x, w, b, 0.0, 0.0, with_scale=True)
    np.testing.assert_array_equal(mean, [1.0])
    np.testing.assert_array_equal(rstd, [1.0])
    np.testing.assert_array_equal(y, [[-0.5, 2.0, -1.5, 2.0]])
    # y_scale = (|x| + |mean|) rstd |w| + |b|
    np.testing.assert_array_equal(ysc, [[1.5, 6.0, 1.5, 6.0]])
    # backward with w = 1, dy = g = [1, 2, 3, 4]: mean(g) = 2.5, mean(g xhat) = 0.5,
    # sum|g|/N = 2.5, sum|g xhat|/N = 2.5
    dy = np.array([[1.0, 2.0, 3.0, 4.0]])
    dx, dw, db, sc = oracle.ln_bwd(x, dy, np.ones(4), 0.0, 0.0, with_scale=True)
    np.testing.assert_array_equal(dx, [[-1.0, -1.0, 1.0, 1.0]])
    np.testing.assert_array_equal(sc, [[6.0, 7.0, 8.0, 9.0]])
    np.testing.assert_array_equal(dw, [-1.0, 2.0, -3.0, 4.0])
    np.testing.assert_array_equal(db, [1.0, 2.0, 3.0, 4.0])
