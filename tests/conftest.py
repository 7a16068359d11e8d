import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def load_build_module():
    """The package's build script, loaded by path so that building does not
    import (and load a stale copy of) the library first."""
    import importlib.util
    path = os.path.join(ROOT, "row_normalization_rmsnorm_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_gb300norm_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def built_package():
    load_build_module().build()
    import row_normalization_rmsnorm_gb300 as pkg
    return pkg


def pytest_terminal_summary(terminalreporter):
    """Summary of the parity checks run in this session: for every output
    checked against the oracle, how many elements passed only through the
    cancellation floor (the n_floor_only count of tests/tolerance.py)."""
    try:
        from tolerance import REPORTS
    except ImportError:
        return
    reps = [r for r in REPORTS if r.get("label")]
    if not reps:
        return
    tr = terminalreporter
    n = sum(r["n"] for r in reps)
    nf = sum(r["n_floor_only"] for r in reps)
    tr.section("parity checks: elements passing only through the cancellation floor")
    tr.write_line(f"{len(reps)} checks, {n} elements, {nf} floor-only ({100.0 * nf / max(n, 1):.4f} %)")
    worst = sorted(reps, key=lambda r: -r["n_floor_only"] / max(r["n"], 1))[:12]
    for r in worst:
        tr.write_line(f"  {r['label'][:60]:60s} n={r['n']:>10d} floor_only={r['n_floor_only']:>7d} "
                      f"({100.0 * r['n_floor_only'] / max(r['n'], 1):.3f} %) rel_l2={r['rel_l2']:.2e}")
