"""Rows split over a thread-block cluster, against the FP64 oracle.

The aligned-row kernels split every row of a cluster into equal column
slices, one per CTA, and add the CTAs' row sums (exchanged through
distributed shared memory) in rank order.  The library does so by itself
where no single CTA takes a row without spilling registers (more than 4096
16-byte chunks, or the per-column state of a wide backward such as the
trainable LayerNorm backward at N = 18432); problems with fewer rows than
SMs keep one CTA per row.  A test hook forces 2, 4 or 8 CTAs per row on any
shape.  Each case below runs every operation, trainable and frozen,
and checks every output element against the oracle, the frozen input
gradient bit for bit against the trainable one, the padding of strided rows,
and dW / dB run to run.
"""
import pytest
import torch

import synthetic_inputs as si
from gpu_util import bits_equal
from test_parity_gpu import check_fadd, check_ln, check_rms, run_fadd, run_ln, run_rms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


@pytest.fixture
def forced(g):
    def set_cluster(c):
        g.norm_debug_tune(5, c)
    yield set_cluster
    g.norm_debug_tune(5, 0)


@pytest.mark.parametrize("M,N", [(1, 4096), (3, 4096), (17, 8192), (128, 4096), (100, 18432), (150, 2048)])
def test_few_rows(g, M, N):
    case = si.norm_case(M, N, seed=41, dtype="bfloat16", gemma=True, fused_add=True)
    check_rms(run_rms(g, case, offset=1.0), case, f"few rows rms {M}x{N}", offset=1.0)
    check_ln(run_ln(g, case), case, f"few rows ln {M}x{N}")
    check_fadd(run_fadd(g, case, offset=1.0), case, f"few rows fadd {M}x{N}", offset=1.0)


@pytest.mark.parametrize("M,N,dtype", [(300, 40960, "bfloat16"), (64, 65536, "bfloat16"),
                                       (40, 20480, "float32"), (33, 65536, "float16")])
def test_wide_rows_split_automatically(g, M, N, dtype):
    case = si.norm_case(M, N, seed=42, dtype=dtype, fused_add=True)
    check_rms(run_rms(g, case, stride=N + 64), case, f"wide rms {dtype} {M}x{N}")
    check_ln(run_ln(g, case, stride=N + 64), case, f"wide ln {dtype} {M}x{N}")
    check_fadd(run_fadd(g, case), case, f"wide fadd {dtype} {M}x{N}")


@pytest.mark.parametrize("c", [2, 4, 8])
def test_forced_cluster_split(g, forced, c):
    forced(c)
    M, N = 1000, 8192
    case = si.norm_case(M, N, seed=43, dtype="bfloat16", fused_add=True)
    check_rms(run_rms(g, case, stride=N + 64), case, f"cluster {c} rms")
    check_ln(run_ln(g, case, dw_dtype=torch.float32), case, f"cluster {c} ln")
    check_fadd(run_fadd(g, case, offset=1.0), case, f"cluster {c} fadd", offset=1.0)
    a = run_ln(g, case, dw_dtype=torch.float32)
    b = run_ln(g, case, dw_dtype=torch.float32)
    assert bits_equal(a["dw"], b["dw"]) and bits_equal(a["db"], b["db"]), "dW/dB differ run to run"
    assert bits_equal(a["dx"].view, b["dx"].view)


@pytest.mark.parametrize("c", [2, 8])
def test_forced_cluster_split_fp32_and_mixed_weights(g, forced, c):
    forced(c)
    for dtype, wdtype in [("float32", "float32"), ("bfloat16", "float32")]:
        case = si.norm_case(257, 4096, seed=44, dtype=dtype, w_dtype=wdtype, outliers=True, fused_add=True)
        check_rms(run_rms(g, case), case, f"cluster {c} rms {dtype}/{wdtype}")
        check_ln(run_ln(g, case), case, f"cluster {c} ln {dtype}/{wdtype}")
        check_fadd(run_fadd(g, case, with_dh=False), case, f"cluster {c} fadd {dtype}/{wdtype}", with_dh=False)


def test_cluster_split_raises_no_device_status(g):
    assert g.norm_device_status(reset=False) == 0
