"""Host-only checks of the C ABI (no GPU needed, no kernel launched).

The library loads, exports every function include/gb300norm.h declares, and
rejects bad arguments on the host with the documented status code before it
touches the device.  Pointers here are fake addresses: every call below fails
validation, so none is ever dereferenced.
"""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gb300norm.h")


@pytest.fixture(scope="module")
def g():
    from conftest import built_package
    return built_package()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GB300NORM_API\s+[\w\s\*]+?\b(norm_\w+)\s*\(", text)))


def test_header_declares_the_six_operations():
    fns = header_functions()
    for name in ["norm_rms_fwd", "norm_rms_bwd", "norm_ln_fwd", "norm_ln_bwd",
                 "norm_fused_add_rms_fwd", "norm_fused_add_rms_bwd", "norm_bwd_workspace_bytes"]:
        assert name in fns


def test_library_exports_every_declared_symbol(g):
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s+(\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name
        assert hasattr(g.lib, name)
    # nothing but the declared C ABI is exported
    assert {e for e in exported if e.startswith("norm_")} == set(header_functions())


def test_binding_covers_exactly_the_header(g):
    assert set(g.SIGNATURES) == set(header_functions())


def test_status_strings_and_version(g):
    for code in range(0, 12):
        s = g.status_str(code)
        assert s and s != "unknown status"
    assert g.status_str(99) == "unknown status"
    assert g.lib.norm_version() >= 10000


# Fake, suitably aligned device addresses; never dereferenced.
X, Y, W, R, DX, DY, WS = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000, 0x60000000, 0x70000000
BF16, F32, F16 = 2, 0, 1


def rms_fwd(g, **kw):
    a = dict(x=X, xs=64, w=W, y=Y, ys=64, rstd=R, M=4, N=64, off=0.0, eps=1e-6, dt=BF16, wdt=BF16)
    a.update(kw)
    return g.lib.norm_rms_fwd(a["x"], a["xs"], a["w"], a["y"], a["ys"], a["rstd"], a["M"], a["N"], a["off"],
                              a["eps"], a["dt"], a["wdt"], None)


def rms_bwd(g, **kw):
    a = dict(dy=DY, dys=64, x=X, xs=64, w=W, rstd=R, dx=DX, dxs=64, dw=None, dwt=F32, ws=None, wsb=0,
             M=4, N=64, off=0.0, eps=1e-6, dt=BF16, wdt=BF16)
    a.update(kw)
    return g.lib.norm_rms_bwd(a["dy"], a["dys"], a["x"], a["xs"], a["w"], a["rstd"], a["dx"], a["dxs"], a["dw"],
                              a["dwt"], a["ws"], a["wsb"], a["M"], a["N"], a["off"], a["eps"], a["dt"], a["wdt"],
                              None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), 1), (dict(y=None), 1), (dict(w=None), 1),
    (dict(M=-1), 2), (dict(N=0), 2), (dict(N=-5), 2), (dict(N=1 << 31), 2),
    (dict(xs=63), 3), (dict(ys=10), 3),
    (dict(dt=F32, wdt=BF16), 4), (dict(dt=F16, wdt=BF16), 4), (dict(dt=7), 4), (dict(wdt=9), 4),
    (dict(x=X + 1), 6), (dict(w=W + 1), 6), (dict(rstd=R + 2), 6),
    (dict(eps=-1e-6), 7), (dict(eps=float("inf")), 7), (dict(off=float("nan")), 7),
    (dict(y=X + 2 * 64, ys=64), 8), (dict(rstd=X + 8), 8), (dict(y=W), 8),
    (dict(M=1 << 40, xs=1 << 30, ys=1 << 30), 2),   # byte extent beyond 63 bits
])
def test_rms_fwd_argument_errors(g, kw, code):
    assert rms_fwd(g, **kw) == code


def test_zero_rows_is_a_host_side_noop(g):
    assert rms_fwd(g, M=0, x=None, y=None, rstd=None) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(dy=None), 1), (dict(dx=None), 1),
    (dict(dw=0x80000000, dwt=F16), 4),            # dw dtype neither f32 nor w dtype
    (dict(dw=0x80000000, ws=None), 5),            # trainable needs a workspace
    (dict(dw=0x80000000, ws=WS + 8, wsb=1 << 30), 5),  # misaligned workspace
    (dict(dx=X), 8),                              # dx may alias dy only
    (dict(dx=DY, dxs=128), 8),                    # same pointer, different stride
])
def test_rms_bwd_argument_errors(g, kw, code):
    assert rms_bwd(g, **kw) == code


def test_ln_bwd_mean_rstd_must_pair(g):
    rc = g.lib.norm_ln_bwd(DY, 64, X, 64, W, 0x90000000, None, DX, 64, None, None, F32, None, 0,
                           4, 64, 0.0, 1e-6, BF16, BF16, None)
    assert rc == 10


def test_fused_add_fwd_outputs_must_not_overlap(g):
    # y and h_out on the same buffer
    rc = g.lib.norm_fused_add_rms_fwd(X, 64, R, 64, W, Y, 64, Y, 64, None, 4, 64, 0.0, 1e-6, BF16, BF16, None)
    assert rc == 8


def test_sum_ranks_argument_errors(g):
    P, O = 0x10000000, 0x20000000   # fake, never dereferenced
    assert g.lib.norm_sum_ranks(P, 0, 64, O, F32, None) == 2          # no rank
    assert g.lib.norm_sum_ranks(P, 2, 0, O, F32, None) == 2           # no column
    assert g.lib.norm_sum_ranks(P, 1 << 31, 64, O, F32, None) == 2    # world above 2^31 - 1
    assert g.lib.norm_sum_ranks(None, 2, 64, O, F32, None) == 1
    assert g.lib.norm_sum_ranks(P, 2, 64, None, F32, None) == 1
    assert g.lib.norm_sum_ranks(P, 2, 64, O, 7, None) == 4
    assert g.lib.norm_sum_ranks(P + 2, 2, 64, O, F32, None) == 6     # parts not 4-byte aligned
    assert g.lib.norm_sum_ranks(P, 2, 64, O + 1, BF16, None) == 6    # out not 2-byte aligned
    assert g.lib.norm_sum_ranks(P, 2, 64, P + 256, F32, None) == 8   # out inside parts


def test_workspace_query_host_paths(g):
    import ctypes
    assert g.lib.norm_bwd_workspace_bytes(4, 64, 1, 0, None) == 1
    out = ctypes.c_size_t(123)
    assert g.lib.norm_bwd_workspace_bytes(-1, 64, 1, 0, ctypes.byref(out)) == 2
    assert g.lib.norm_bwd_workspace_bytes(8, 64, 0, 0, ctypes.byref(out)) == 0 and out.value == 0
    assert g.lib.norm_bwd_workspace_bytes(0, 64, 1, 1, ctypes.byref(out)) == 0 and out.value == 0


def test_debug_tune_keys_and_range(g):
    # keys 1..4 accept 0..64 (0 = automatic), key 5 (CTAs per row) 0, 1, 2,
    # 4 or 8, key 6 (withhold each row group's last copy) 0 or 1, and leave
    # the library in its automatic state again; anything else is
    # NORM_ERR_ARG (10)
    for key in (1, 2, 3, 4):
        assert g.lib.norm_debug_tune(key, 64) == 0
        assert g.lib.norm_debug_tune(key, 0) == 0
    for v in (1, 2, 4, 8, 0):
        assert g.lib.norm_debug_tune(5, v) == 0
    for v in (3, 16, 64, -1):
        assert g.lib.norm_debug_tune(5, v) == 10
    assert g.lib.norm_debug_tune(6, 1) == 0
    assert g.lib.norm_debug_tune(6, 0) == 0
    assert g.lib.norm_debug_tune(6, 2) == 10
    assert g.lib.norm_debug_tune(0, 1) == 10
    assert g.lib.norm_debug_tune(7, 1) == 10
    assert g.lib.norm_debug_tune(4, -1) == 10
    assert g.lib.norm_debug_tune(4, 65) == 10


def test_binding_rejects_cpu_tensors(g):
    import torch
    x = torch.zeros(2, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        g.norm_rms_fwd(x, torch.ones(8, dtype=torch.bfloat16), torch.empty_like(x))


def test_oracle_is_not_reachable_from_the_product_package():
    pkg = os.path.join(ROOT, "row_normalization_rmsnorm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                for needle in ("import oracle", "from oracle", "libnormoracle", "norm_oracle"):
                    assert needle not in text, (f, needle)
