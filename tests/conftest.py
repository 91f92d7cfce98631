import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")
    config.addinivalue_line("markers", "big: full-size workload (several GB of device memory)")


@pytest.fixture(scope="session")
def lsc():
    """The C-ABI binding; loading fails loudly if liblsc.so is missing."""
    from linear_attention_state_lsc_gb300 import lsc as binding
    binding.load()
    return binding
