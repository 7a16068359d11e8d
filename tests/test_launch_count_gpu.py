"""Kernels per call, counted by the library itself (norm_debug_launches: one
count per successful kernel launch, the only way this library launches).

A frozen backward is one kernel -- the row kernel with every weight-gradient
instruction compiled out, and no column reduce ("perf(norm): skip dW/dB
calculation when parameters are frozen", Key Changes); a trainable backward
is the row kernel and the column reduce; a forward is one kernel; an empty
trainable backward (M = 0) is the column reduce alone (dW / dB set to zero).
"""
import pytest
import torch

import synthetic_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def launches(g, fn):
    g.norm_debug_launches(reset=True)
    fn()
    torch.cuda.synchronize()
    return g.norm_debug_launches(reset=True)


@pytest.mark.parametrize("M,N", [(512, 4096), (33, 1001), (100, 40960)])   # staged, general, cluster split
def test_kernels_per_call(g, M, N):
    c = si.norm_case(M, N, seed=95, dtype="bfloat16", fused_add=True)
    d = {k: v.cuda() for k, v in c.items()}
    e = lambda: torch.empty(M, N, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    f = lambda n: torch.empty(n, dtype=torch.float32, device="cuda")  # noqa: E731
    ws = torch.empty(max(16, g.norm_bwd_workspace_bytes(M, N, True, True)), dtype=torch.uint8, device="cuda")
    y, h, dx, rstd, mean, dw, db = e(), e(), e(), f(M), f(M), f(N), f(N)
    calls = {
        "rms_fwd": (lambda: g.norm_rms_fwd(d["x"], d["w"], y, rstd), 1),
        "rms_bwd": (lambda: g.norm_rms_bwd(d["dy"], d["x"], d["w"], rstd, dx, dw, ws), 2),
        "rms_bwd_frozen": (lambda: g.norm_rms_bwd(d["dy"], d["x"], d["w"], rstd, dx), 1),
        "ln_fwd": (lambda: g.norm_ln_fwd(d["x"], d["w"], d["b"], y, mean, rstd), 1),
        "ln_bwd": (lambda: g.norm_ln_bwd(d["dy"], d["x"], d["w"], mean, rstd, dx, dw, db, ws), 2),
        "ln_bwd_db_only": (lambda: g.norm_ln_bwd(d["dy"], d["x"], d["w"], mean, rstd, dx, None, db, ws), 2),
        "ln_bwd_frozen": (lambda: g.norm_ln_bwd(d["dy"], d["x"], d["w"], mean, rstd, dx), 1),
        "fadd_fwd": (lambda: g.norm_fused_add_rms_fwd(d["x"], d["residual"], d["w"], y, h, rstd), 1),
        "fadd_bwd": (lambda: g.norm_fused_add_rms_bwd(d["dy"], d["dh_out"], h, d["w"], rstd, dx, dw, ws), 2),
        "fadd_bwd_frozen": (lambda: g.norm_fused_add_rms_bwd(d["dy"], d["dh_out"], h, d["w"], rstd, dx), 1),
    }
    for name, (fn, want) in calls.items():
        assert launches(g, fn) == want, name
    assert g.norm_device_status(reset=False) == 0


def test_empty_and_argument_errors(g):
    N = 4096
    x = torch.empty(0, N, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((N,), float("nan"), device="cuda")
    r = torch.empty(0, device="cuda")
    assert launches(g, lambda: g.norm_rms_fwd(x, w, x, r)) == 0                       # M = 0: nothing
    assert launches(g, lambda: g.norm_rms_bwd(x, x, w, r, x)) == 0                    # frozen, M = 0
    assert launches(g, lambda: g.norm_rms_bwd(x, x, w, r, x, dw,
                                              torch.empty(16, dtype=torch.uint8, device="cuda"))) == 1
    assert bool((dw == 0).all())                                                       # dW of no rows
    # a refused call enqueues nothing
    with pytest.raises(Exception):
        g.norm_rms_fwd(torch.empty(4, N, dtype=torch.bfloat16, device="cuda"), w[:N - 1],
                       torch.empty(4, N, dtype=torch.bfloat16, device="cuda"))
    assert g.norm_debug_launches(reset=True) == 0
