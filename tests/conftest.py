import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def golden_path(name: str) -> str:
    return os.path.join(ROOT, "tests", "golden", name)


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA-path library, built in-tree if needed (no GPU needed to load it)."""
    from paged_kv_decode_v2_gb300 import build as pkg_build
    pkg_build.build()
    import paged_kv_decode_v2_gb300 as pa
    return pa
