import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload parity (minutes)")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def kda():
    """The CUDA binding; builds libkda.so first when it is missing or stale."""
    from linear_attention_03_gb300 import build
    build.build()
    from linear_attention_03_gb300 import kda as mod
    return mod
