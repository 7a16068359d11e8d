"""Concurrent callers: host threads, each on its own CUDA stream, calling the
library at once.

The ctypes binding releases the interpreter lock during each C call, so the
calls below really overlap on the host -- the device query, the launch-shape
caches (occupancy, kernel attributes, cluster fits) and the launches -- and
their kernels may overlap on the GPU.  Every thread owns its tensors and
workspace.  Each call's outputs must equal, bit for bit, those of the same
call made alone on the default stream first (a launch shape depends only on
the device and the problem, never on the stream or on timing).
"""
import threading

import pytest
import torch

import synthetic_inputs as si
from gpu_util import bits_equal

pytestmark = pytest.mark.gpu

# staged (4 and 2 chunks per thread, exact and not), a cluster split, the
# general kernel
SHAPES = [(777, 4096), (513, 8192), (1000, 1536), (300, 2560), (64, 18432), (129, 1001)]


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def job(g, M, N, seed):
    """Every operation (trainable backward) on one shape; returns the
    outputs as a list."""
    c = si.norm_case(M, N, seed=seed, dtype="bfloat16", fused_add=True)
    d = {k: v.cuda() for k, v in c.items()}
    e = lambda: torch.empty(M, N, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    f = lambda n: torch.empty(n, dtype=torch.float32, device="cuda")  # noqa: E731
    ws = torch.empty(max(16, g.norm_bwd_workspace_bytes(M, N, True, True)), dtype=torch.uint8, device="cuda")

    def run():
        y, rstd, dx, dw = e(), f(M), e(), f(N)
        g.norm_rms_fwd(d["x"], d["w"], y, rstd, 1.0, 1e-6)
        g.norm_rms_bwd(d["dy"], d["x"], d["w"], rstd, dx, dw, ws, 1.0, 1e-6)
        ly, mean, lrstd, ldx, ldw, ldb = e(), f(M), f(M), e(), f(N), f(N)
        g.norm_ln_fwd(d["x"], d["w"], d["b"], ly, mean, lrstd, 0.0, 1e-6)
        g.norm_ln_bwd(d["dy"], d["x"], d["w"], mean, lrstd, ldx, ldw, ldb, ws, 0.0, 1e-6)
        fy, fh, frstd, fdx, fdw = e(), e(), f(M), e(), f(N)
        g.norm_fused_add_rms_fwd(d["x"], d["residual"], d["w"], fy, fh, frstd, 0.0, 1e-6)
        g.norm_fused_add_rms_bwd(d["dy"], d["dh_out"], fh, d["w"], frstd, fdx, fdw, ws, 0.0, 1e-6)
        return [y, rstd, dx, dw, ly, mean, lrstd, ldx, ldw, ldb, fy, fh, frstd, fdx, fdw]
    return run


def test_threads_on_their_own_streams_get_the_bits_of_a_lone_call(g):
    runs = [job(g, M, N, 200 + i) for i, (M, N) in enumerate(SHAPES)]
    ref = []
    for run in runs:
        ref.append([t.clone() for t in run()])
    torch.cuda.synchronize()

    for rep in range(3):
        results = [None] * len(runs)
        errors = []
        start = threading.Barrier(len(runs))

        def worker(i):
            try:
                s = torch.cuda.Stream()
                start.wait()
                with torch.cuda.stream(s):
                    out = runs[i]()
                s.synchronize()
                results[i] = out
            except Exception as exc:   # reported below, on the main thread
                errors.append((i, repr(exc)))

        threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(runs))]
        for t in threads:
            t.start()
        for t in threads:
            t.join(timeout=120)
        assert not errors, errors
        for i, (M, N) in enumerate(SHAPES):
            assert results[i] is not None, f"thread {i} did not finish"
            for k, (a, b) in enumerate(zip(results[i], ref[i])):
                assert bits_equal(a, b), f"rep {rep}, {M}x{N}, output {k} differs from the lone call"
    assert g.norm_device_status(reset=False) == 0
