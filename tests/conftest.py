import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True


@pytest.fixture(scope="session")
def fge(cuda_ok):
    """The built binding on a CUDA device (builds libfge.so in-tree if needed)."""
    from fp8_grouped_expert_gb300 import build as _build
    _build.build()
    import fp8_grouped_expert_gb300 as mod
    mod.lib()
    return mod
