import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionstart(session):
    # Build the CUDA library in-tree (and the C oracle) when nvcc is present,
    # so a fresh checkout can run the suite; nothing here falls back to a
    # CPU path if the build is missing.
    if shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc"):
        from cast_transpose_gb300 import _build
        _build.build()
    import oracle
    oracle.build()


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.lib()
    return oracle
