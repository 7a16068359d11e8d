"""Multi-rank host logic on CPU (gloo, world size 2): row sharding, the
max-over-ranks timing and the fixed-order dW combine of an M-sharded
backward, checked against the single-process oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synthetic_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _dist_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_gb300norm_dist", os.path.join(ROOT, "row_normalization_rmsnorm_gb300", "dist.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


@pytest.mark.parametrize("M", [0, 1, 7, 8192, 8193])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_rows_partition(M, world):
    d = _dist_module()
    ranges = [d.shard_rows(M, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == M
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = _dist_module()
        M = 37
        r0, r1 = d.shard_rows(M, rank, world)
        res = {}
        # each rank's column sums over its own rows (the oracle standing in for
        # the library's FP32 column reduction), combined in rank order
        c = si.norm_case(M, 24, seed=9, dtype="float32", with_bias=False)
        x, dy, w = (c[k].double().numpy() for k in ("x", "dy", "w"))
        _, dw_part, _ = oracle.rms_bwd(x[r0:r1], dy[r0:r1], w, 0.0, 1e-6)
        res["rms_dw"] = d.combine_partials(torch.from_numpy(dw_part)).numpy().tolist()
        c = si.norm_case(M, 24, seed=10, dtype="float32")
        x, dy, w = (c[k].double().numpy() for k in ("x", "dy", "w"))
        _, dw_part, db_part, _ = oracle.ln_bwd(x[r0:r1], dy[r0:r1], w, 0.0, 1e-6)
        res["ln_dw"] = d.combine_partials(torch.from_numpy(dw_part)).numpy().tolist()
        out_db = torch.empty(24, dtype=torch.float64)
        res["ln_db"] = d.combine_into(torch.from_numpy(db_part), out_db).numpy().tolist()
        c = si.norm_case(M, 24, seed=11, dtype="float32", with_bias=False, fused_add=True)
        h, dy, w, dh = (c[k].double().numpy() for k in ("x", "dy", "w", "dh_out"))
        _, dw_part, _ = oracle.fused_add_rms_bwd(h[r0:r1], dy[r0:r1], w, dh[r0:r1], 1.0, 1e-6)
        res["fadd_dw"] = d.combine_partials(torch.from_numpy(dw_part)).numpy().tolist()
        res["t"] = d.max_over_ranks(10.0 + rank)
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_sharded_backward_combines_to_the_single_process_gradients():
    import oracle
    oracle.build()
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    M = 37
    c = si.norm_case(M, 24, seed=9, dtype="float32", with_bias=False)
    x, dy, w = (c[k].double().numpy() for k in ("x", "dy", "w"))
    ref = {"rms_dw": oracle.rms_bwd(x, dy, w, 0.0, 1e-6)[1]}
    c = si.norm_case(M, 24, seed=10, dtype="float32")
    x, dy, w = (c[k].double().numpy() for k in ("x", "dy", "w"))
    _, ref["ln_dw"], ref["ln_db"], _ = oracle.ln_bwd(x, dy, w, 0.0, 1e-6)
    c = si.norm_case(M, 24, seed=11, dtype="float32", with_bias=False, fused_add=True)
    h, dy, w, dh = (c[k].double().numpy() for k in ("x", "dy", "w", "dh_out"))
    ref["fadd_dw"] = oracle.fused_add_rms_bwd(h, dy, w, dh, 1.0, 1e-6)[1]
    for key, r in ref.items():
        assert out[0][key] == out[1][key], key      # same bits on every rank
        np.testing.assert_allclose(out[0][key], r, rtol=1e-13, atol=1e-13, err_msg=key)
    assert out[0]["t"] == out[1]["t"] == 11.0       # max over ranks
