import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (large-shape parity)")


@pytest.fixture(scope="session")
def lib():
    """The loaded C-ABI library (skips when absent on a CPU-only machine)."""
    from newton_schulz_gb300 import binding
    try:
        return binding.load()
    except OSError as e:  # pragma: no cover - only when not built
        pytest.skip(f"libmuon not built: {e}")


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True
