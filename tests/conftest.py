import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); parity tests through the C ABI")


def build_library():
    """Build (if stale) libtgemm.so via the standalone build script."""
    import importlib.util
    path = os.path.join(ROOT, "tiled_dense_gemm_02_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("tgemm_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()
