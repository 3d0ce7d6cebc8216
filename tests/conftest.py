import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: large workload (seconds to minutes)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The product's ctypes binding, built in-tree if needed. Fails loudly if it cannot load."""
    import bwd_situ_glu_gb300 as sg
    sg.build()
    sg.load()
    return sg
