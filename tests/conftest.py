import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(params=["two_pass", "online"])
def decode_kernel(request, monkeypatch):
    """Both decode kernels behind every decode entry point, each forced: the
    two-pass split kernel and the single-pass online-softmax one (the library
    otherwise picks one per call from the split length)."""
    monkeypatch.setenv("FORGE_DECODE_KERNEL", request.param)
    return request.param
