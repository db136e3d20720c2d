"""Shared pytest set-up: markers and import paths.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on a CPU-only host.
"""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled sm_103a library")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def w4lib():
    """Build (if stale) and load the CUDA library; GPU tests only.

    Skips when this host has no CUDA device.  On a GPU host a missing or
    broken library is an error, never a skip."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device on this host")
    from w4a16_weight_only_gemm_gb300 import _native, build
    build.build()
    return _native.lib()
