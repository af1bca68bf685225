import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def _gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree on first use."""
    from invariant_paged_prefill_gb300 import _lib, build
    if not os.path.exists(build.library_path()):
        build.build_library()
    return _lib.load()


@pytest.fixture(scope="session")
def cuda():
    if not _gpu_available():
        pytest.skip("no CUDA device")
    import torch
    return torch.device("cuda:0")
