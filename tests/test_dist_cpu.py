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
        case = si.norm_case(37, 24, seed=9, dtype="float32", with_bias=False)
        x, dy, w = (case[k].double().numpy() for k in ("x", "dy", "w"))
        r0, r1 = d.shard_rows(37, rank, world)
        _, dw_part, _ = oracle.rms_bwd(x[r0:r1], dy[r0:r1], w, 0.0, 1e-6)
        total = d.combine_partials(torch.from_numpy(dw_part))
        t = d.max_over_ranks(10.0 + rank)
        out[rank] = (total.numpy().tolist(), t)
    finally:
        dist.destroy_process_group()


def test_sharded_backward_combines_to_the_single_process_dw():
    import oracle
    oracle.build()
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    case = si.norm_case(37, 24, seed=9, dtype="float32", with_bias=False)
    x, dy, w = (case[k].double().numpy() for k in ("x", "dy", "w"))
    _, dw_full, _ = oracle.rms_bwd(x, dy, w, 0.0, 1e-6)
    got0, t0 = out[0]
    got1, t1 = out[1]
    assert got0 == got1                        # same bits on every rank
    np.testing.assert_allclose(got0, dw_full, rtol=1e-13, atol=1e-13)
    assert t0 == t1 == 11.0                    # max over ranks
