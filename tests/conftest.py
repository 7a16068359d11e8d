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
