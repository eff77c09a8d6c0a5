import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running (minutes); full-size workloads")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def cuda():
    """The CUDA binding; a GPU test fails (does not skip) when the library cannot be loaded."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_rule_gb300 as kda
    kda.load()
    return kda
