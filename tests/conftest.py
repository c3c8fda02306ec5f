"""Shared pytest set-up: the gpu marker, and building the CPU oracle.

Tests marked gpu need a CUDA device and the compiled library; everything else
runs on the CPU (oracle pins, host-side validation, ABI symbol checks).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled libufp4")


@pytest.fixture(scope="session")
def oracle():
    from oracle import oracle as o
    o.lib()
    return o
