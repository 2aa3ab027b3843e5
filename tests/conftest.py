"""Shared pytest set-up: repo root on sys.path and the ``gpu`` marker."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built library's binding, on a GPU; checks the device status word
    before and after the session (a bounded wait that gave up fails it)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device: the gpu tests need a GB300")
    from moe_finalize_rmsnorm_gb300.build import build
    build()
    import moe_finalize_rmsnorm_gb300 as mf
    assert mf.device_status(clear=True) == 0
    yield mf
    assert mf.device_status(clear=True) == 0, "a kernel's bounded wait timed out"
