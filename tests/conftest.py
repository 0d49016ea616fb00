import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library through its Python binding; the binding raises if the
    shared object is missing, so GPU tests never run on a fallback."""
    import lossless_draft_verification_gb300 as specv
    from lossless_draft_verification_gb300 import build
    build.build()
    specv.load()
    return specv
