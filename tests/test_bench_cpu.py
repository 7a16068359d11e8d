"""Host-side checks of bench.py (no GPU): the reference arm's JSON line, the
algorithmic byte counts behind every GB/s figure, the shape grid, and the
source hash that guards committed ncu counters."""
import json
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes_at_8192():
    # reads of x, dy, residual, w (and bias), rstd (and mean), writes of y,
    # dx, h_out and dW (dB) -- bf16 tensors, FP32 statistics
    M = N = 8192
    MN = M * N
    assert bench.op_bytes("rms_fwd", M, N) == 2 * MN * 2 + N * 2 + 4 * M == 268484608
    assert bench.op_bytes("ln_fwd", M, N) == 2 * MN * 2 + 2 * N * 2 + 8 * M == 268533760
    assert bench.op_bytes("fadd_fwd", M, N) == 4 * MN * 2 + N * 2 + 4 * M == 536920064
    assert bench.op_bytes("rms_bwd", M, N) == 402718720
    assert bench.op_bytes("rms_bwd", M, N, trainable=False) == 402718720 - N * 2
    assert bench.op_bytes("ln_bwd", M, N) == 402767872
    assert bench.op_bytes("ln_bwd", M, N, trainable=False) == 402767872 - 2 * N * 2
    assert bench.op_bytes("fadd_bwd", M, N) == 536936448
    with pytest.raises(ValueError):
        bench.op_bytes("softmax", M, N)


def test_grid_covers_the_configured_shapes():
    fams = bench.grid_families()
    for sh in bench.GRID_SHAPES:
        assert {"rms", "ln"} <= set(fams[sh])
    for sh in bench.FADD_SHAPES + [(8192, 8192)]:
        assert "fadd" in fams[sh]
    for sh in bench.GEMMA_SHAPES:
        assert "rms" in fams[sh]
    assert all(len(set(v)) == len(v) for v in fams.values())   # no family twice


def test_source_hash_ignores_comments(tmp_path):
    src = os.path.join(ROOT, "row_normalization_rmsnorm_gb300", "csrc")
    pkg = tmp_path / "row_normalization_rmsnorm_gb300"
    shutil.copytree(src, pkg / "csrc")
    old_root = bench.ROOT
    try:
        bench.ROOT = str(tmp_path)
        h0 = bench.kernel_source_hash()
        f = pkg / "csrc" / "colreduce.cu"
        text = f.read_text()
        f.write_text("// a comment line\n" + text.replace("\n\n", "\n\n/* a block\n comment */\n", 1))
        assert bench.kernel_source_hash() == h0
        f.write_text(text.replace("kCrClusterRows = 512", "kCrClusterRows = 513"))
        assert bench.kernel_source_hash() != h0
    finally:
        bench.ROOT = old_root


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1", "--M", "64", "--N", "512", "--ref-rows", "16"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["metric"] == bench.METRIC and j["unit"] == "GB/s" and j["higher_is_better"] is True
    assert j["steps"] == 2 and j["warmup"] == 1 and j["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_baseline_runs_on_every_core_and_keeps_the_single_thread_figure():
    host = bench.host_inputs(64, 512, seed=0)
    cb = bench.cpu_baseline(host, target_s=0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s"
    assert cb["cores"] == bench.host_cores() >= 1
    assert cb["value"] > 0 and cb["single_thread_value"] > 0
    assert f"on {cb['cores']} threads" in cb["sample"]


def test_parallel_oracle_blocks_partition_the_sample():
    # the row blocks cover the sample exactly once, in order, and the block
    # partial sums of dW add up (in block order) to the one-block result
    import numpy as np
    host = bench.host_inputs(40, 256, seed=1)
    one, w, lb = bench.oracle_blocks(host, 40, 1)
    many, _, _ = bench.oracle_blocks(host, 40, 6)
    assert sum(b["rx"].shape[0] for b in many) == 40
    np.testing.assert_array_equal(np.concatenate([b["lx"] for b in many]), one[0]["lx"])
    ref = bench.oracle_block(one[0], w, lb)
    parts = [bench.oracle_block(b, w, lb) for b in many]
    for k in range(4):
        tot = parts[0][k].copy()
        for p in parts[1:]:
            tot += p[k]
        np.testing.assert_allclose(tot, ref[k], rtol=1e-12, atol=1e-12)


def test_e2e_upload_dependencies_cover_every_reader():
    # the e2e pipeline's next upload into a tensor waits for every kernel that
    # reads it; each operation's host inputs must be listed with their readers
    for op in bench.OPS:
        for k in bench.Workload.IN[op]:
            assert op in bench.Workload.READERS[k], (op, k)
    # a forward's activations and weights are read again by its backward
    assert "rms_bwd" in bench.Workload.READERS["rms.x"] and "ln_bwd" in bench.Workload.READERS["ln.x"]
    assert "fadd_bwd" in bench.Workload.READERS["fadd.w"]


def test_launch_count_claim():
    # the bench's gpu_launches claim: one row kernel per call, plus the column
    # reduce of a trainable backward, plus (sharded over ranks) one rank-order
    # sum per gradient
    assert [bench.launches_per_op(op) for op in bench.OPS] == [1, 1, 1, 2, 2, 2]
    assert [bench.launches_per_op(op, trainable=False) for op in bench.OPS] == [1] * 6
    assert [bench.launches_per_op(op, world=2) for op in bench.OPS] == [1, 1, 1, 3, 4, 3]


def test_committed_traffic_covers_every_operation_at_the_large_shapes():
    import csv
    rows = list(csv.DictReader(open(os.path.join(ROOT, "profiles", "ncu_traffic_shapes.csv"))))
    shapes = {(int(r["M"]), int(r["N"])) for r in rows}
    assert {(4096, 4096), (4096, 8192), (8192, 4096), (8192, 8192), (32768, 8192)} <= shapes
    for M, N in shapes:
        ops = {r["op"] for r in rows if (int(r["M"]), int(r["N"])) == (M, N)}
        assert ops == set(bench.OPS)
    for r in rows:
        # inputs read once, outputs written once: the total stays within the
        # partial rows' few percent of the algorithmic bytes
        assert 0.98 < float(r["ratio"]) < 1.12, r
