import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _ensure_library():
    """Build libew.so (and the oracle) once if a compiler is present and the
    library is missing, so the host-side ABI tests run on a fresh checkout."""
    import shutil
    lib = os.path.join(ROOT, "memory_bound_elementwise_gb300", "_lib", "libew.so")
    if os.path.exists(lib) or not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        return
    from memory_bound_elementwise_gb300 import _build
    _build.build()


def pytest_configure(config):
    _ensure_library()
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test, skipped unless EW_SLOW_TESTS=1")


def pytest_collection_modifyitems(config, items):
    if os.environ.get("EW_SLOW_TESTS") == "1":
        return
    skip = pytest.mark.skip(reason="slow; set EW_SLOW_TESTS=1")
    for item in items:
        if "slow" in item.keywords:
            item.add_marker(skip)
