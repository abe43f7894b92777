import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); parity against the CPU oracle")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session", autouse=True)
def _built():
    """Compile the C generator and oracle (gcc, seconds) before any test; the CUDA library is built on
    demand by the tests that load it."""
    import oracle
    import synth
    synth.build()
    oracle.build()
    yield
