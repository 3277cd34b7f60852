import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")
    config.addinivalue_line("markers", "slow: long-running CPU check")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def ensure_built():
    """Build libtpconv.so and the C oracle if they are missing (nvcc/gcc)."""
    import importlib.util
    lib = os.path.join(ROOT, "equivariant_gnn_tensor_gb300", "libtpconv.so")
    spec = importlib.util.spec_from_file_location("_tpconv_build", os.path.join(ROOT, "equivariant_gnn_tensor_gb300",
                                                                                 "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    from oracle import cref
    cref.build()
    return lib


@pytest.fixture(scope="session")
def tpc():
    ensure_built()
    import equivariant_gnn_tensor_gb300 as m
    return m
