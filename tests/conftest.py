import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")


def pytest_collection_modifyitems(config, items):
    # GPU tests need the CUDA runtime; without one they are skipped rather than
    # silently routed anywhere else.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def _built_library():
    """Compile libtrfn.so (nvcc cross-compiles without a GPU) and the oracle
    before any test runs; a failure to build fails the session loudly."""
    from image_preprocessing_gb300.build import build_library
    from oracle.build import build_oracle
    build_library()
    build_oracle()
    yield
