"""The backward workspace contract, on both forms of the column reduce (the
scalar one, fewer than 512 partial rows, and the 8-CTA cluster one):
  * dW / dB and dx are bit-identical whether the workspace is 128-byte
    aligned or only 16-byte aligned, and whatever it held before (a second
    call on the same workspace gives the same bits);
  * the bytes of the buffer before and after the workspace keep their
    contents;
  * on an aligned workspace the results match the FP64 oracle
    (test_parity_gpu's checks).
"""
import pytest
import torch

import synthetic_inputs as si
from gpu_util import bits_equal
from test_parity_gpu import check_ln, check_rms

pytestmark = pytest.mark.gpu

GUARD = 4096   # bytes of sentinel before and after the workspace


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def guarded(g, M, N, shift):
    """A workspace of the size the call needs, `shift` bytes past a
    128-byte aligned point of a larger buffer filled with 0xA5."""
    need = g.norm_bwd_workspace_bytes(M, N, True, True)
    buf = torch.full((GUARD + need + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    assert buf.data_ptr() % 256 == 0
    ws = buf[GUARD + shift:GUARD + shift + need]
    return buf, ws, need


def guards_intact(buf, shift, need):
    lo = buf[:GUARD + shift]
    hi = buf[GUARD + shift + need:]
    return bool((lo == 0xA5).all()) and bool((hi == 0xA5).all())


def ln_grads(g, case, ws):
    x, dy, w, b = (case[k].cuda() for k in ("x", "dy", "w", "b"))
    M, N = x.shape
    y, dx = torch.empty_like(x), torch.empty_like(x)
    mean = torch.empty(M, dtype=torch.float32, device="cuda")
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    dw = torch.empty(N, dtype=torch.float32, device="cuda")
    db = torch.empty(N, dtype=torch.float32, device="cuda")
    g.norm_ln_fwd(x, w, b, y, mean, rstd)
    g.norm_ln_bwd(dy, x, w, mean, rstd, dx, dw, db, ws)
    torch.cuda.synchronize()
    return dw, db, dx


# (M, N): 8192 columns with few partial rows (scalar reduce); 4096 columns
# with many rows (cluster reduce at >= 512 partial rows); 1024 x 96 (N % 32
# == 0, a ragged last column block of the cluster form's 128-column tiles)
@pytest.mark.parametrize("M,N", [(2048, 8192), (20000, 4096), (30000, 96)])
def test_workspace_alignment_and_reuse(g, M, N):
    case = si.norm_case(M, N, seed=61, dtype="bfloat16")
    results = {}
    for shift in (0, 16):   # 128-byte aligned, then 16-byte aligned
        buf, ws, need = guarded(g, M, N, shift)
        a = ln_grads(g, case, ws)
        b = ln_grads(g, case, ws)   # the same workspace again
        assert guards_intact(buf, shift, need), f"bytes outside the workspace changed (shift {shift})"
        assert all(bits_equal(u, v) for u, v in zip(a, b)), f"second call differs (shift {shift})"
        results[shift] = a
    for u, v in zip(results[0], results[16]):
        assert bits_equal(u, v), "the workspace alignment changed dW / dB / dx"
    assert g.norm_device_status(reset=False) == 0


def test_aligned_workspace_against_oracle(g):
    # the parity helpers allocate 256-byte aligned workspaces
    M, N = 3000, 8192
    case = si.norm_case(M, N, seed=62, dtype="bfloat16", gemma=True)
    from test_parity_gpu import run_ln, run_rms
    check_rms(run_rms(g, case, offset=1.0), case, "workspace rms", offset=1.0)
    check_ln(run_ln(g, case, dw_dtype=torch.float32), case, "workspace ln")
    assert g.norm_device_status(reset=False) == 0
