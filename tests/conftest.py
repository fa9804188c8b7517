import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: large shapes; minutes of CPU oracle time")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library binding; GPU tests fail loudly if it cannot be loaded."""
    import fp8_block_scaled_bias_b300 as m
    return m
