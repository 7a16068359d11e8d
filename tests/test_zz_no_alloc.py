"""The no-allocation RMSNorm backward (norm_rms_bwd_noalloc) against the
workspace version (norm_rms_bwd), through the C ABI.

norm_rms_bwd_noalloc serves callers that cannot allocate device memory: it
keeps the dW partial sums in the library's fixed scratch array instead of a
caller-provided workspace.  It runs the same kernels with the same launch
shape as the workspace version, so two calls in a row (different inputs)
must give bit-identical dx and dW; the second is also checked against the
FP64 oracle.  A problem too large for the scratch is refused before anything
runs.  This file is collected last so
that a stop at its first failure has already run every other test.
"""
import pytest
import torch

import synthetic_inputs as si
import oracle
from gpu_util import bits_equal, dw_scale, f64, unit_xhat, workspace
from tolerance import check, check_dw, dtype_name

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def run_both(g, case, dw_dtype, offset):
    x, dy, w = (case[k].cuda() for k in ("x", "dy", "w"))
    M, N = x.shape
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    g.norm_rms_fwd(x, w, y, rstd, offset, 1e-6)
    dx_ws, dx_na = torch.empty_like(x), torch.empty_like(x)
    dw_ws = torch.full((N,), float("nan"), dtype=dw_dtype, device="cuda")
    dw_na = torch.full((N,), float("nan"), dtype=dw_dtype, device="cuda")
    g.norm_rms_bwd(dy, x, w, rstd, dx_ws, dw_ws, workspace(g, M, N, True), offset, 1e-6)
    g.norm_rms_bwd_noalloc(dy, x, w, rstd, dx_na, dw_na, offset, 1e-6)
    torch.cuda.synchronize()
    return dx_ws, dw_ws, dx_na, dw_na


def test_noalloc_matches_workspace_version_twice(g):
    cases = [(si.norm_case(8192, 8192, seed=11, dtype="bfloat16", with_bias=False), torch.bfloat16, 0.0),
             (si.norm_case(1000, 4096, seed=12, dtype="bfloat16", gemma=True, with_bias=False), torch.float32, 1.0)]
    assert g.lib.norm_noalloc_scratch_bytes() >= g.norm_bwd_workspace_bytes(8192, 8192, True)
    for case, dw_dtype, offset in cases:
        dx_ws, dw_ws, dx_na, dw_na = run_both(g, case, dw_dtype, offset)
        assert bits_equal(dx_na, dx_ws), "noalloc dx differs from the workspace call"
        assert bits_equal(dw_na, dw_ws), "noalloc dW differs from the workspace call"
    # the last call against the oracle (saved-rstd path, as the GPU used its forward's rstd)
    x, dy, w = (f64(case[k]) for k in ("x", "dy", "w"))
    rstd = oracle.rms_fwd(x, w, offset, 1e-6)[1]
    dxr, dwr, sc = oracle.rms_bwd(x, dy, w, offset, 1e-6, with_scale=True, rstd=rstd)
    check(dx_na, dxr, dtype_name(dx_na), scale=sc, label="noalloc dx vs oracle")
    check_dw(dw_na, dwr, dtype_name(dw_na), dw_scale(dy, unit_xhat(x, False, 1e-6)), label="noalloc dw vs oracle")


def test_noalloc_refuses_a_problem_larger_than_its_scratch(g):
    M, N = 8192, 65536
    assert g.norm_bwd_workspace_bytes(M, N, True) > g.lib.norm_noalloc_scratch_bytes()
    x = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(M, dtype=torch.float32, device="cuda")
    dx = torch.empty_like(x)
    dw = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.NormError) as e:
        g.norm_rms_bwd_noalloc(x, x, w, rstd, dx, dw)
    assert e.value.status == 11
