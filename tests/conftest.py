import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size configurations (minutes)")


@pytest.fixture(scope="session", autouse=True)
def _host_libraries():
    """The CPU-side libraries every test needs: the input generator and the oracle (gcc, seconds)."""
    import oracle
    import synth

    synth.build()
    oracle.build()
    yield


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def q8():
    """The CUDA library's Python binding, built for sm_103a on first use; GPU tests only."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import moe_add_rmsnorm_gb300 as m
    return m
