"""Failure detection: a row copy that never lands ends the kernel with an
error status, not a hang.

Every wait of the aligned-row kernels is bounded (2 s, then the device
status word is set and the kernel returns).  A test hook (norm_debug_tune
key 6) makes each row group's producer withhold the copy of its last row:
the consumers' wait for that row runs out, the kernel skips that row's
outputs and returns, and -- because the withheld row is the last, so every
copy that was issued has been waited for -- no copy is left in flight when
a CTA exits.  Each case checks that the status word reports the timeout,
clears it, and then runs the same call without the hook against the FP64
oracle: the context stays usable.  No GPU fault, trap or endless wait is
involved.
"""
import time

import pytest
import torch

import synthetic_inputs as si
from test_parity_gpu import check_ln, check_rms, run_ln, run_rms

pytestmark = pytest.mark.gpu

KEY_HOLD_LAST, KEY_CLUSTER = 6, 5
STATUS_WAIT_TIMEOUT = 1


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def withheld(g, fn):
    """Run fn with the last-row copies withheld; return (device status,
    seconds) and leave the hook off and the status cleared."""
    assert g.norm_device_status(reset=True) == 0
    g.norm_debug_tune(KEY_HOLD_LAST, 1)
    try:
        t0 = time.perf_counter()
        fn()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        g.norm_debug_tune(KEY_HOLD_LAST, 0)
    return g.norm_device_status(reset=True), dt


@pytest.mark.parametrize("op", ["rms", "ln"])
def test_forward_and_backward_report_a_wait_that_ran_out(g, op):
    M, N = 600, 4096
    case = si.norm_case(M, N, seed=81, dtype="bfloat16")
    run, check = (run_rms, check_rms) if op == "rms" else (run_ln, check_ln)
    status, dt = withheld(g, lambda: run(g, case))
    assert status & STATUS_WAIT_TIMEOUT, f"{op}: no timeout reported (status {status})"
    assert dt >= 1.5, f"{op}: the bounded wait should take about 2 s, took {dt:.2f} s"
    check(run(g, case), case, f"{op} after a timeout")
    assert g.norm_device_status(reset=False) == 0


def test_cluster_split_reports_a_wait_that_ran_out(g):
    # every CTA of a cluster gives up on the same row, then all meet at the
    # cluster barrier on the way out
    M, N = 256, 8192
    case = si.norm_case(M, N, seed=82, dtype="bfloat16")
    g.norm_debug_tune(KEY_CLUSTER, 2)
    try:
        status, _ = withheld(g, lambda: run_ln(g, case))
        assert status & STATUS_WAIT_TIMEOUT
        check_ln(run_ln(g, case), case, "cluster ln after a timeout")
    finally:
        g.norm_debug_tune(KEY_CLUSTER, 0)
    assert g.norm_device_status(reset=False) == 0


def test_one_row_per_group_withholds_every_copy(g):
    # M below the row-group count: each group has one row and issues no copy
    M, N = 40, 8192
    case = si.norm_case(M, N, seed=83, dtype="bfloat16")
    status, _ = withheld(g, lambda: run_rms(g, case))
    assert status & STATUS_WAIT_TIMEOUT
    check_rms(run_rms(g, case), case, "rms after a timeout")
