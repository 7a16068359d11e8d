"""The staged kernels' copy ring and launch shapes, forced through the test
hook, against the FP64 oracle.

Each CTA streams its rows through a ring of S shared-memory stages filled by
bulk copies S-1 rows ahead; a stage is refilled once every thread is done
with the row it held, and the mbarrier phase of each stage flips on every
reuse.  Here the ring is forced to its minimum depth (2 stages; 3 for the
LayerNorm forward, which holds two rows), with one CTA per SM so that each
CTA walks many rows and every stage is reused many times, and every
chunks-per-thread shape (1, 2, 4, 8) is forced in turn.  Every output is
checked against the oracle and the frozen input gradient against the
trainable one, bit for bit; no wait may run out (device status 0).
"""
import pytest

import synthetic_inputs as si
from test_parity_gpu import check_fadd, check_ln, check_rms, run_fadd, run_ln, run_rms

pytestmark = pytest.mark.gpu

KEY_NPT, KEY_CTAS, KEY_STAGES = 1, 2, 3


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


@pytest.fixture
def tune(g):
    keys = []

    def set_(key, value):
        keys.append(key)
        g.norm_debug_tune(key, value)
    yield set_
    for k in keys:
        g.norm_debug_tune(k, 0)


@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("npt", [1, 2, 4, 8])
def test_minimum_ring_depth_and_every_chunk_shape(g, tune, stages, npt):
    tune(KEY_STAGES, stages)
    tune(KEY_CTAS, 1)
    tune(KEY_NPT, npt)
    M, N = 3001, 4096   # about 20 rows per CTA, a ragged last round
    case = si.norm_case(M, N, seed=51, dtype="bfloat16", gemma=True, fused_add=True)
    label = f"ring S={stages} npt={npt}"
    check_rms(run_rms(g, case, offset=1.0), case, f"{label} rms", offset=1.0)
    check_ln(run_ln(g, case), case, f"{label} ln")
    check_fadd(run_fadd(g, case, offset=1.0), case, f"{label} fadd", offset=1.0)
    assert g.norm_device_status(reset=False) == 0


@pytest.mark.parametrize("ctas", [2, 8])
def test_several_ctas_per_sm_at_minimum_depth(g, tune, ctas):
    tune(KEY_STAGES, 2)
    tune(KEY_CTAS, ctas)
    M, N = 2500, 2048
    case = si.norm_case(M, N, seed=52, dtype="bfloat16", fused_add=True)
    check_rms(run_rms(g, case, stride=N + 64), case, f"ctas={ctas} rms")
    check_ln(run_ln(g, case, stride=N + 64), case, f"ctas={ctas} ln")
    check_fadd(run_fadd(g, case), case, f"ctas={ctas} fadd")
    assert g.norm_device_status(reset=False) == 0
