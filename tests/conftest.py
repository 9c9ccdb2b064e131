import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The C-ABI library, built in-tree if missing (no GPU needed to load it)."""
    from speculative_decode_gateddeltanet_gb300 import build as pkg_build

    pkg_build.build()
    from speculative_decode_gateddeltanet_gb300 import gdn

    return gdn
