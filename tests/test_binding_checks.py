"""The Python binding checks every buffer's extent before calling the C ABI.

The C entry points receive only pointers, M, N and dtype codes, so a short
weight, a 16-bit output given with an FP32 input or a stats vector with too
few rows would make a kernel read or write out of bounds.  Each case below
builds one such mismatch from CPU tensors: the binding must raise ValueError
(shape / dtype checks run before the device check), and a call whose shapes
are all right must get as far as the device check (TypeError for a CPU
tensor).  No kernel is launched.
"""
import contextlib

import pytest
import torch

M, N = 4, 64
BF, F32, F16 = torch.bfloat16, torch.float32, torch.float16


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def mat(dt=BF, m=M, n=N):
    return torch.zeros(m, n, dtype=dt)


def vec(n=N, dt=BF):
    return torch.ones(n, dtype=dt)


def good_args(op):
    """A complete, consistent argument set per wrapper (CPU tensors)."""
    if op == "rms_fwd":
        return dict(x=mat(), w=vec(), y=mat(), rstd=vec(M, F32))
    if op == "rms_bwd":
        return dict(dy=mat(), x=mat(), w=vec(), rstd=vec(M, F32), dx=mat(), dw=vec(N, F32),
                    workspace=torch.empty(16, dtype=torch.uint8))
    if op == "ln_fwd":
        return dict(x=mat(), w=vec(), b=vec(), y=mat(), mean=vec(M, F32), rstd=vec(M, F32))
    if op == "ln_bwd":
        return dict(dy=mat(), x=mat(), w=vec(), mean=vec(M, F32), rstd=vec(M, F32), dx=mat(), dw=vec(),
                    db=vec(), workspace=torch.empty(16, dtype=torch.uint8))
    if op == "fadd_fwd":
        return dict(x=mat(), residual=mat(), w=vec(), y=mat(), h_out=mat(), rstd=vec(M, F32))
    if op == "fadd_bwd":
        return dict(dy=mat(), dh_out=mat(), h=mat(), w=vec(), rstd=vec(M, F32), dx=mat(), dw=vec(N, F32),
                    workspace=torch.empty(16, dtype=torch.uint8))
    if op == "rms_bwd_noalloc":
        return dict(dy=mat(), x=mat(), w=vec(), rstd=vec(M, F32), dx=mat(), dw=vec(N, F32))
    raise ValueError(op)


def call(g, op, a):
    fn = {"rms_fwd": g.norm_rms_fwd, "rms_bwd": g.norm_rms_bwd, "ln_fwd": g.norm_ln_fwd,
          "ln_bwd": g.norm_ln_bwd, "fadd_fwd": g.norm_fused_add_rms_fwd, "fadd_bwd": g.norm_fused_add_rms_bwd,
          "rms_bwd_noalloc": g.norm_rms_bwd_noalloc}[op]
    return fn(**a)


# (operation, argument, replacement): each replacement breaks one extent or dtype
BAD = [
    ("rms_fwd", "w", vec(N - 1)), ("rms_fwd", "w", mat()), ("rms_fwd", "y", mat(F32)),
    ("rms_fwd", "y", mat(n=N - 1)), ("rms_fwd", "y", mat(m=M + 1)), ("rms_fwd", "rstd", vec(M - 1, F32)),
    ("rms_fwd", "rstd", vec(M, BF)), ("rms_fwd", "x", torch.zeros(M, N, 1, dtype=BF)),
    ("rms_fwd", "x", mat(torch.float64)), ("rms_fwd", "w", vec(N, torch.float64)),
    ("rms_bwd", "dy", mat(m=M - 1)), ("rms_bwd", "dx", mat(F16)), ("rms_bwd", "dw", vec(N - 8, F32)),
    ("rms_bwd", "dw", vec(N, F16)), ("rms_bwd", "rstd", vec(M - 1, F32)),
    ("ln_fwd", "b", vec(N - 1)), ("ln_fwd", "b", vec(N, F32)), ("ln_fwd", "mean", vec(M - 1, F32)),
    ("ln_fwd", "y", mat(n=2 * N)),
    ("ln_bwd", "db", vec(N - 1)), ("ln_bwd", "db", vec(N, F32)),   # dw bf16, db f32: one dW/dB dtype
    ("ln_bwd", "mean", vec(M - 2, F32)), ("ln_bwd", "dy", mat(F32)),
    ("fadd_fwd", "residual", mat(m=M - 1)), ("fadd_fwd", "h_out", mat(F16)), ("fadd_fwd", "y", mat(n=N + 8)),
    ("fadd_bwd", "dh_out", mat(n=N - 1)), ("fadd_bwd", "dy", mat(m=2)), ("fadd_bwd", "dx", mat(F32)),
    ("fadd_bwd", "dw", vec(2 * N, F32)),
    ("rms_bwd_noalloc", "dw", vec(N + 1, F32)), ("rms_bwd_noalloc", "dx", mat(m=M + 3)),
]


@pytest.mark.parametrize("op,arg,bad", BAD, ids=[f"{o}-{a}-{i}" for i, (o, a, _) in enumerate(BAD)])
def test_mismatched_buffer_is_refused_before_any_launch(g, op, arg, bad):
    a = good_args(op)
    a[arg] = bad
    with pytest.raises(ValueError):
        call(g, op, a)


def test_noncontiguous_rows_are_refused(g):
    a = good_args("rms_fwd")
    a["y"] = torch.zeros(N, M, dtype=BF).t()
    with pytest.raises(ValueError):
        call(g, "rms_fwd", a)


@pytest.mark.parametrize("op", ["rms_fwd", "rms_bwd", "ln_fwd", "ln_bwd", "fadd_fwd", "fadd_bwd",
                                "rms_bwd_noalloc"])
def test_consistent_arguments_reach_the_device_check(g, op):
    # every extent is right: the only error left is that the tensors are on the CPU
    with pytest.raises(TypeError):
        call(g, op, good_args(op))


def test_calls_run_with_the_tensors_device_current(g, monkeypatch):
    # The C ABI takes launch shapes and its status word from the current
    # device; a call on tensors of another device switches to it first.
    from row_normalization_rmsnorm_gb300 import _binding as B
    switched = []

    @contextlib.contextmanager
    def fake_device(dev):
        switched.append(dev)
        yield

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "device", fake_device)
    assert B._on(0, lambda: "same") == "same" and switched == []
    assert B._on(3, lambda: "other") == "other" and switched == [3]


@pytest.mark.parametrize("parts,out,err", [
    (torch.zeros(3, N), torch.zeros(N), TypeError),                 # consistent: reaches the device check
    (torch.zeros(N), torch.zeros(N), ValueError),                   # parts not 2-D
    (torch.zeros(0, N), torch.zeros(N), ValueError),                # no rank
    (torch.zeros(3, N, dtype=BF), torch.zeros(N), ValueError),      # parts not FP32
    (torch.zeros(N, 3).t(), torch.zeros(N), ValueError),            # parts not contiguous
    (torch.zeros(3, N), torch.zeros(N - 1), ValueError),            # out too short
    (torch.zeros(3, N), torch.zeros(N, dtype=torch.int32), ValueError),   # out dtype
])
def test_sum_ranks_checks(g, parts, out, err):
    with pytest.raises(err):
        g.norm_sum_ranks(parts, out)
