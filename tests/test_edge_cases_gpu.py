"""Edge cases of the CUDA path, each against the FP64 oracle or against the
same library's other route to the same result."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_util import Strided, bits_equal, f64, workspace
from test_parity_gpu import (EPS, check_fadd, check_ln, check_rms, run_fadd, run_ln, run_rms)
from tolerance import check, check_dw, dtype_name, rounded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


@pytest.fixture
def loop_path(g):
    g.norm_debug_set_path(2)
    yield
    g.norm_debug_set_path(0)


# ---------------------------------------------------------------------------
# sizes
# ---------------------------------------------------------------------------

def test_zero_rows(g):
    N = 64
    x = torch.empty(0, N, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    g.norm_rms_fwd(x, w, torch.empty_like(x), torch.empty(0, device="cuda"))
    dw = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    g.norm_rms_bwd(x, x, w, torch.empty(0, device="cuda"), torch.empty_like(x), dw, None)
    db = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    dw2 = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    g.norm_ln_bwd(x, x, w, None, None, torch.empty_like(x), dw2, db, None)
    torch.cuda.synchronize()
    assert bool((dw == 0).all()) and bool((dw2 == 0).all()) and bool((db == 0).all())


@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 9, 33, 100, 129])
@pytest.mark.parametrize("M", [1, 5])
@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
def test_tiny_rows(g, M, N, dtype):
    case = si.norm_case(M, N, seed=N, dtype=dtype)
    check_rms(run_rms(g, case), case, f"tiny rms {M}x{N} {dtype}")
    if N > 1:   # a one-element row has zero variance: LayerNorm output is the bias
        check_ln(run_ln(g, case), case, f"tiny ln {M}x{N} {dtype}")


def hard_rows(N, gen):
    """Rows against the forward's one-pass statistics (each thread's sums
    about one of its own elements, merged exactly), FP64: [well-conditioned
    ones], [ones whose mean is 1e5 / 5e4 times their spread]."""
    good = []
    r = torch.randn(N, generator=gen, dtype=torch.float64)
    r[::4] = 1e4          # the first element of every 16-byte fp32 chunk: every thread's shift
    good.append(r)
    r = torch.randn(N, generator=gen, dtype=torch.float64)
    r[0] = 1e4            # one outlier, thread 0's shift
    good.append(r)
    good.append(torch.full((N,), 3.0, dtype=torch.float64))   # zero variance
    offset = [1000.0 + 0.01 * torch.randn(N, generator=gen, dtype=torch.float64),
              -50.0 + 1e-3 * torch.randn(N, generator=gen, dtype=torch.float64)]
    return good, offset


@pytest.mark.parametrize("N", [4096, 8192])
def test_layernorm_statistics_hard_rows(g, N):
    """FP32 rows built against the forward's one-pass statistics, against the
    two-pass FP64 oracle.  mean and rstd are checked on every row.  y, dx, dW
    and dB are checked on the well-conditioned ones.  Where |mean| / spread is
    1e5, y itself carries the FP32 rounding of the mean, which any FP32
    statistics share."""
    gen = torch.Generator().manual_seed(5)
    good, offset = hard_rows(N, gen)
    x_all = torch.stack(good + offset).repeat(32, 1).to(torch.float32)
    M = x_all.shape[0]
    w = (1 + 0.1 * torch.randn(N, generator=gen)).to(torch.float32)
    b = (0.1 * torch.randn(N, generator=gen)).to(torch.float32)
    xd = x_all.cuda()
    y = torch.empty_like(xd)
    mean = torch.empty(M, device="cuda")
    rstd = torch.empty(M, device="cuda")
    g.norm_ln_fwd(xd, w.cuda(), b.cuda(), y, mean, rstd, 0.0, EPS)
    _, ref_mean, ref_rstd, _ = oracle.ln_fwd(f64(x_all), f64(w), f64(b), 0.0, EPS)
    check(mean, ref_mean, "float32", scale=16 * np.abs(f64(x_all)).mean(axis=1), label=f"hard rows mean N={N}")
    check(rstd, ref_rstd, "float32", label=f"hard rows rstd N={N}")
    xg = torch.stack(good).repeat(64, 1).to(torch.float32)
    case = {"x": xg, "dy": torch.randn(xg.shape[0], N, generator=gen).to(torch.float32), "w": w, "b": b}
    check_ln(run_ln(g, case), case, f"hard rows ln fp32 N={N}")


def test_single_element_layernorm_gives_bias(g):
    case = si.norm_case(4, 1, seed=1, dtype="float32")
    out = run_ln(g, case)
    np.testing.assert_array_equal(out["y"].view.cpu().numpy()[:, 0], case["b"].numpy()[0])


def test_wide_rows_general_kernel(g):
    case = si.norm_case(3, 65537, seed=2, dtype="bfloat16")
    check_rms(run_rms(g, case), case, "rms 3x65537")
    check_ln(run_ln(g, case), case, "ln 3x65537")


def test_many_narrow_rows(g):
    case = si.norm_case(100000, 64, seed=3, dtype="bfloat16")
    check_rms(run_rms(g, case), case, "rms 100000x64")
    check_ln(run_ln(g, case), case, "ln 100000x64")


# ---------------------------------------------------------------------------
# alignment and kernel families
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("lead", [1, 2, 3, 5, 7])
def test_unaligned_row_starts(g, lead):
    case = si.norm_case(64, 4096, seed=lead, dtype="bfloat16", fused_add=True)
    check_rms(run_rms(g, case, lead=lead), case, f"rms lead {lead}")
    check_ln(run_ln(g, case, lead=lead), case, f"ln lead {lead}")


@pytest.mark.parametrize("M,N", [(512, 4096), (256, 8192)])
def test_general_kernel_matches_oracle_on_aligned_rows(g, loop_path, M, N):
    case = si.norm_case(M, N, seed=4, dtype="bfloat16", fused_add=True)
    check_rms(run_rms(g, case), case, "loop rms")
    check_ln(run_ln(g, case), case, "loop ln")
    check_fadd(run_fadd(g, case), case, "loop fadd")


def test_kernel_families_agree(g):
    case = si.norm_case(300, 8192, seed=5, dtype="bfloat16")
    staged = run_rms(g, case)
    g.norm_debug_set_path(2)
    try:
        loop = run_rms(g, case)
    finally:
        g.norm_debug_set_path(0)
    a = staged["dx"].view.float()
    b = loop["dx"].view.float()
    # both round the same FP32 formula; they may differ by one bf16 ulp
    assert float((a - b).abs().max()) <= float(a.abs().max()) * 2 ** -7
    assert bits_equal(staged["y"].view, loop["y"].view) or \
        float((staged["y"].view.float() - loop["y"].view.float()).abs().max()) <= 2 ** -6


@pytest.mark.parametrize("dtype,wdtype", [("float16", "float32"), ("float32", "float32"), ("float16", "float16")])
def test_other_dtypes_on_the_staged_kernel(g, dtype, wdtype):
    case = si.norm_case(257, 8192, seed=6, dtype=dtype, w_dtype=wdtype, fused_add=True)
    check_rms(run_rms(g, case), case, f"rms {dtype}/{wdtype}")
    check_ln(run_ln(g, case), case, f"ln {dtype}/{wdtype}")
    check_fadd(run_fadd(g, case), case, f"fadd {dtype}/{wdtype}")


# ---------------------------------------------------------------------------
# in place and recomputed statistics
# ---------------------------------------------------------------------------

def test_in_place_calls_match_out_of_place(g):
    M, N = 333, 8192
    case = si.norm_case(M, N, seed=7, dtype="bfloat16", fused_add=True)
    d = {k: v.cuda() for k, v in case.items()}
    rstd = torch.empty(M, device="cuda")
    # RMSNorm forward, y == x
    y = torch.empty_like(d["x"])
    g.norm_rms_fwd(d["x"], d["w"], y, rstd)
    xi = d["x"].clone()
    g.norm_rms_fwd(xi, d["w"], xi, rstd)
    assert bits_equal(xi, y)
    # LayerNorm forward, y == x
    mean = torch.empty(M, device="cuda")
    g.norm_ln_fwd(d["x"], d["w"], d["b"], y, mean, rstd)
    xi = d["x"].clone()
    g.norm_ln_fwd(xi, d["w"], d["b"], xi, mean, rstd)
    assert bits_equal(xi, y)
    # RMSNorm backward, dx == dy
    g.norm_rms_fwd(d["x"], d["w"], y, rstd)
    dx = torch.empty_like(d["x"])
    g.norm_rms_bwd(d["dy"], d["x"], d["w"], rstd, dx)
    dyi = d["dy"].clone()
    g.norm_rms_bwd(dyi, d["x"], d["w"], rstd, dyi)
    assert bits_equal(dyi, dx)
    # FusedAdd forward, h_out == residual; backward, dx == dh_out
    h = torch.empty_like(d["x"])
    g.norm_fused_add_rms_fwd(d["x"], d["residual"], d["w"], y, h, rstd)
    ri = d["residual"].clone()
    y2 = torch.empty_like(y)
    g.norm_fused_add_rms_fwd(d["x"], ri, d["w"], y2, ri, rstd)
    assert bits_equal(ri, h) and bits_equal(y2, y)
    g.norm_fused_add_rms_bwd(d["dy"], d["dh_out"], h, d["w"], rstd, dx)
    dhi = d["dh_out"].clone()
    g.norm_fused_add_rms_bwd(d["dy"], dhi, h, d["w"], rstd, dhi)
    torch.cuda.synchronize()
    assert bits_equal(dhi, dx)


@pytest.mark.parametrize("N", [4096, 4095])
def test_backward_recomputes_statistics(g, N):
    M = 200
    case = si.norm_case(M, N, seed=8, dtype="bfloat16")
    x, dy, w = (case[k].cuda() for k in ("x", "dy", "w"))
    x64, dy64, w64 = f64(case["x"]), f64(case["dy"]), f64(case["w"])
    dx = torch.empty_like(x)
    g.norm_rms_bwd(dy, x, w, None, dx)
    ref, _, sc = oracle.rms_bwd(x64, dy64, w64, 0.0, EPS, with_scale=True)
    check(dx, ref, "bfloat16", scale=sc, label="rms bwd recomputed rstd")
    g.norm_ln_bwd(dy, x, w, None, None, dx)
    ref, _, _, sc = oracle.ln_bwd(x64, dy64, w64, 0.0, EPS, with_scale=True)
    torch.cuda.synchronize()
    check(dx, ref, "bfloat16", scale=sc, label="ln bwd recomputed stats")


# ---------------------------------------------------------------------------
# determinism, streams, graphs
# ---------------------------------------------------------------------------

def test_weight_gradients_are_deterministic(g):
    M, N = 4096, 8192
    case = si.norm_case(M, N, seed=9, dtype="bfloat16")
    a = run_ln(g, case, dw_dtype=torch.float32)
    b = run_ln(g, case, dw_dtype=torch.float32)
    assert bits_equal(a["dw"], b["dw"]) and bits_equal(a["db"], b["db"])
    c = run_rms(g, case, dw_dtype=torch.float32)
    e = run_rms(g, case, dw_dtype=torch.float32)
    assert bits_equal(c["dw"], e["dw"])


@pytest.mark.parametrize("M,N", [(8192, 4096), (4096, 64), (8192, 2052), (4096, 4095)])
def test_many_partial_rows_column_reduce(g, M, N):
    """Trainable backwards that leave 512 or more dW partial rows take the
    thread-block-cluster column reduce when N % 4 == 0: 608 rows at N = 4096,
    1216 at N = 64 (one partial 128-column tile) and at N = 2052 (a ragged
    last tile).  N = 4095 (general row kernel, partial rows not 16-byte
    aligned) keeps the scalar reduce.  dW and dB match the oracle and repeat
    bit for bit."""
    case = si.norm_case(M, N, seed=31, dtype="bfloat16")
    a = run_rms(g, case, dw_dtype=torch.float32)
    check_rms(a, case, f"cluster reduce rms {M}x{N}")
    b = run_rms(g, case, dw_dtype=torch.float32)
    assert bits_equal(a["dw"], b["dw"])
    c = run_fadd(g, si.norm_case(M, N, seed=32, dtype="bfloat16", with_bias=False, fused_add=True),
                 dw_dtype=torch.bfloat16)
    e = run_fadd(g, si.norm_case(M, N, seed=32, dtype="bfloat16", with_bias=False, fused_add=True),
                 dw_dtype=torch.bfloat16)
    assert bits_equal(c["dw"], e["dw"])
    ln1 = run_ln(g, case, dw_dtype=torch.float32)
    check_ln(ln1, case, f"cluster reduce ln {M}x{N}")
    ln2 = run_ln(g, case, dw_dtype=torch.float32)
    assert bits_equal(ln1["dw"], ln2["dw"]) and bits_equal(ln1["db"], ln2["db"])


def test_non_default_stream(g):
    M, N = 1024, 4096
    case = si.norm_case(M, N, seed=10, dtype="bfloat16")
    x, dy, w = (case[k].cuda() for k in ("x", "dy", "w"))
    s = torch.cuda.Stream()
    y, dx = torch.empty_like(x), torch.empty_like(x)
    rstd = torch.empty(M, device="cuda")
    dw = torch.empty(N, dtype=torch.float32, device="cuda")
    ws = workspace(g, M, N, True)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.norm_rms_fwd(x, w, y, rstd)
        g.norm_rms_bwd(dy, x, w, rstd, dx, dw, ws)
    s.synchronize()
    ref_y, _ = oracle.rms_fwd(f64(case["x"]), f64(case["w"]), 0.0, EPS)
    check(y, ref_y, "bfloat16", label="stream y")
    ref_dx, ref_dw, sc = oracle.rms_bwd(f64(case["x"]), f64(case["dy"]), f64(case["w"]), 0.0, EPS,
                                        with_scale=True)
    check(dx, ref_dx, "bfloat16", scale=sc, label="stream dx")


def test_cuda_graph_replay_with_changed_inputs(g):
    """Capture forward + trainable backward once, then replay after writing
    new x, w and dy into the captured buffers ([B] diagnostics: CUDA Graph
    replay with changed X, W and dY)."""
    M, N = 2048, 4096
    cases = [si.norm_case(M, N, seed=s, dtype="bfloat16", gemma=True, with_bias=False) for s in (20, 21)]
    x = cases[0]["x"].cuda()
    dy = cases[0]["dy"].cuda()
    w = cases[0]["w"].cuda()
    y, dx = torch.empty_like(x), torch.empty_like(x)
    rstd = torch.empty(M, device="cuda")
    dw = torch.empty(N, dtype=torch.float32, device="cuda")
    ws = workspace(g, M, N, True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):      # warm-up outside capture (first-use setup)
        g.norm_rms_fwd(x, w, y, rstd, 1.0)
        g.norm_rms_bwd(dy, x, w, rstd, dx, dw, ws, 1.0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.norm_rms_fwd(x, w, y, rstd, 1.0)
        g.norm_rms_bwd(dy, x, w, rstd, dx, dw, ws, 1.0)
    for case in cases[::-1] + cases:
        x.copy_(case["x"])
        dy.copy_(case["dy"])
        w.copy_(case["w"])
        graph.replay()
        torch.cuda.synchronize()
        x64, dy64, w64 = f64(case["x"]), f64(case["dy"]), f64(case["w"])
        ry, rr = oracle.rms_fwd(x64, w64, 1.0, EPS)
        rdx, rdw, sc = oracle.rms_bwd(x64, dy64, w64, 1.0, EPS, with_scale=True, rstd=rr)
        check(y, ry, "bfloat16", label="graph y")
        check(dx, rdx, "bfloat16", scale=sc, label="graph dx")
        xh = oracle.rms_fwd(x64, np.ones(N), 0.0, EPS)[0]
        check_dw(dw, rdw, "float32", np.abs(dy64 * xh).sum(0), label="graph dw")


# ---------------------------------------------------------------------------
# errors that need the device's size
# ---------------------------------------------------------------------------

def test_workspace_one_byte_short_is_refused(g):
    M, N = 1024, 4096
    x = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    nb = g.norm_bwd_workspace_bytes(M, N, True)
    assert nb > 0 and g.norm_bwd_workspace_bytes(M, N, False, False) == 0
    ws = torch.empty(nb - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.NormError) as e:
        g.norm_rms_bwd(x, x, w, None, torch.empty_like(x), torch.empty(N, device="cuda"), ws)
    assert e.value.status == 5


def test_device_status_is_clear(g):
    assert g.norm_device_status(reset=False) == 0


# ---------------------------------------------------------------------------
# LayerNorm with a weight offset and without a bias
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N", [(1000, 4096), (300, 8192), (257, 4097), (128, 18432)])
@pytest.mark.parametrize("offset,bias", [(1.0, True), (1.0, False), (0.0, False)])
def test_layernorm_offset_and_no_bias(g, M, N, offset, bias):
    """The weight offset (W' = w + offset, formed in FP32) is not LayerNorm's
    usual form but the ABI takes it for every operation; with it, and with
    no bias, LayerNorm forward and backward (trainable and frozen) match the
    oracle on the staged kernel (4096, 8192), the general kernel (4097) and
    the cluster split (18432 at 128 rows)."""
    case = si.norm_case(M, N, seed=71, dtype="bfloat16", gemma=offset != 0.0, with_bias=bias)
    label = f"ln {M}x{N} offset {offset} bias {bias}"
    check_ln(run_ln(g, case, offset=offset, bias=bias), case, label, offset=offset, bias=bias)
    assert g.norm_device_status(reset=False) == 0


@pytest.mark.parametrize("M,N", [(1000, 1536), (700, 2560), (300, 3072), (200, 5120), (64, 12288)])
def test_model_widths(g, M, N):
    """Hidden sizes of common models that are not powers of two: the launch
    rule picks chunks per thread by how exactly the threads cover a row (2
    chunks at 1536 and 2560, 4 from 3072 up); every operation against the
    oracle, Gemma offset on RMSNorm and FusedAdd."""
    case = si.norm_case(M, N, seed=91, dtype="bfloat16", gemma=True, fused_add=True)
    check_rms(run_rms(g, case, offset=1.0), case, f"rms {M}x{N}", offset=1.0)
    check_ln(run_ln(g, case), case, f"ln {M}x{N}")
    check_fadd(run_fadd(g, case, offset=1.0), case, f"fadd {M}x{N}", offset=1.0)
    assert g.norm_device_status(reset=False) == 0


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
def test_every_small_width_and_alignment(g, dtype):
    """Every row width N = 2..64 with every base offset of 0..7 elements
    (bf16: 16-byte aligned only at offset 0 and N % 8 == 0, so nearly every
    case takes the general kernel and the rest the staged one), RMSNorm and
    LayerNorm forward and backward, trainable and frozen, against the oracle
    -- with NaN sentinels before and after every buffer that must stay
    untouched (checked inside check_rms / check_ln)."""
    for N in range(2, 65):
        case = si.norm_case(3, N, seed=1000 + N, dtype=dtype)
        for lead in range(8):
            check_rms(run_rms(g, case, lead=lead), case, f"rms N={N} lead={lead} {dtype}")
            check_ln(run_ln(g, case, lead=lead), case, f"ln N={N} lead={lead} {dtype}")
    assert g.norm_device_status(reset=False) == 0
