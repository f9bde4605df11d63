"""Shared pytest set-up: the ``gpu`` marker and the repository root on sys.path."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def gpu_lib():
    """libmrn.so built for sm_103a and loaded; skips when no CUDA device is visible."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dual_epsilon_sandwich_gb300 import _build, mrn
    _build.build()
    return mrn.lib()
