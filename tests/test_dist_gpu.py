"""The M-sharded backward (row_normalization_rmsnorm_gb300.dist) on one GPU.

With one process the exchange is the identity, so sharded_backward must give
the bits of the plain call.  Two ranks are then played one after the other
on this GPU (each shard's backward runs alone; nothing waits on another
rank): each shard's FP32 column sums, added in rank order, must match the
oracle's gradient of the whole problem.  The multi-process exchange itself
is covered on CPU with gloo ranks (tests/test_dist_cpu.py).  The exchange's
sum over ranks (norm_sum_ranks) is checked bit for bit against its
definition: FP32 additions in rank order, then one rounding to the output
type.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_util import bits_equal, dw_scale, f64, unit_xhat, workspace
from tolerance import check_dw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def test_single_rank_sharded_backward_is_the_plain_call(g):
    from row_normalization_rmsnorm_gb300 import dist as gd
    M, N = 1000, 4096
    c = si.norm_case(M, N, seed=31, dtype="bfloat16")
    x, dy, w = (c[k].cuda() for k in ("x", "dy", "w"))
    mean, rstd = torch.empty(M, device="cuda"), torch.empty(M, device="cuda")
    g.norm_ln_fwd(x, w, c["b"].cuda(), torch.empty_like(x), mean, rstd)
    ws = workspace(g, M, N, True, True)
    dx0, dx1 = torch.empty_like(x), torch.empty_like(x)
    dw0, db0 = torch.empty_like(w), torch.empty_like(w)
    dw1, db1 = torch.empty_like(w), torch.empty_like(w)
    p0, p1 = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    g.norm_ln_bwd(dy, x, w, mean, rstd, dx0, p0, p1, ws)
    dw0.copy_(p0), db0.copy_(p1)
    gd.sharded_backward("ln", dy, x, w, (mean, rstd), dx1, dw1, db1, workspace=ws)
    torch.cuda.synchronize()
    assert bits_equal(dx0, dx1) and bits_equal(dw0, dw1) and bits_equal(db0, db1)


@pytest.mark.parametrize("kind", ["rms", "ln", "fadd"])
def test_two_shards_added_in_rank_order_match_the_oracle(g, kind):
    from row_normalization_rmsnorm_gb300 import dist as gd
    M, N, world = 1537, 2048, 2
    c = si.norm_case(M, N, seed=32, dtype="bfloat16", fused_add=True)
    x, dy, w, dh = (c[k].cuda() for k in ("x", "dy", "w", "dh_out"))
    parts_w, parts_b = [], []
    for rank in range(world):
        r0, r1 = gd.shard_rows(M, rank, world)
        xs, dys, dhs = x[r0:r1], dy[r0:r1], dh[r0:r1]
        m = r1 - r0
        rstd, mean = torch.empty(m, device="cuda"), torch.empty(m, device="cuda")
        dx = torch.empty_like(xs)
        pw = torch.empty(N, device="cuda")
        pb = torch.empty(N, device="cuda") if kind == "ln" else None
        ws = workspace(g, m, N, True, kind == "ln")
        if kind == "rms":
            g.norm_rms_fwd(xs, w, torch.empty_like(xs), rstd)
            gd.sharded_backward("rms", dys, xs, w, rstd, dx, pw, workspace=ws)
        elif kind == "ln":
            g.norm_ln_fwd(xs, w, c["b"].cuda(), torch.empty_like(xs), mean, rstd)
            gd.sharded_backward("ln", dys, xs, w, (mean, rstd), dx, pw, pb, workspace=ws)
        else:
            gd.sharded_backward("fadd", dys, xs, w, None, dx, pw, dh_out=dhs, workspace=ws)
        parts_w.append(pw)
        parts_b.append(pb)
    # the exchange step: the shards' FP32 sums added in rank order (the
    # library's kernel, as sharded_backward runs it after its all-gather)
    tot_w = torch.empty(N, device="cuda")
    g.norm_sum_ranks(torch.stack(parts_w), tot_w)
    torch.cuda.synchronize()
    x64, dy64, w64, dh64 = f64(c["x"]), f64(c["dy"]), f64(c["w"]), f64(c["dh_out"])
    if kind == "rms":
        _, ref, _ = oracle.rms_bwd(x64, dy64, w64, 0.0, 1e-6)
    elif kind == "ln":
        _, ref, refb, _ = oracle.ln_bwd(x64, dy64, w64, 0.0, 1e-6)
        tot_b = torch.empty(N, device="cuda")
        g.norm_sum_ranks(torch.stack(parts_b), tot_b)
        check_dw(tot_b, refb, "float32", np.abs(dy64).sum(0), label="two shards ln db")
    else:
        _, ref, _ = oracle.fused_add_rms_bwd(x64, dy64, w64, dh64, 0.0, 1e-6)
    check_dw(tot_w, ref, "float32", dw_scale(dy64, unit_xhat(x64, kind == "ln", 1e-6)),
             label=f"two shards {kind} dw")


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("N", [1, 777, 8192])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_sum_ranks_is_the_rank_order_fp32_sum(g, world, N, out_dtype):
    gen = torch.Generator().manual_seed(world * 100003 + N)
    # magnitudes spread over many binades, so a different order of the
    # additions would change the bits
    parts = (torch.randn(world, N, generator=gen) * torch.exp2(torch.randint(-12, 12, (world, N), generator=gen))
             ).float()
    ref = parts[0].numpy().copy()
    for r in range(1, world):
        ref = (ref + parts[r].numpy()).astype(np.float32)   # one FP32 rounding per addition
    ref = torch.from_numpy(ref).to(out_dtype)               # converted once (round to nearest even)
    out = torch.full((N,), float("nan"), dtype=out_dtype, device="cuda")
    g.norm_sum_ranks(parts.cuda(), out)
    torch.cuda.synchronize()
    assert bits_equal(out.cpu(), ref)


def test_combine_on_one_rank_converts_once(g):
    from row_normalization_rmsnorm_gb300 import dist as gd
    p = torch.randn(4096, device="cuda") * 3
    out = torch.empty(4096, dtype=torch.bfloat16, device="cuda")
    gd.combine_into(p, out)
    torch.cuda.synchronize()
    assert bits_equal(out.cpu(), p.cpu().to(torch.bfloat16))
    assert gd.combine_into(p, p) is p   # FP32 on one rank: the partial is the result
