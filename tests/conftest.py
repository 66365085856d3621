import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size oracle work (minutes of CPU)")


@pytest.fixture(scope="session")
def mb():
    """The C-ABI binding, with libmb.so built (compiled on first use)."""
    from mixed_prefill_decode_gb300 import build, binding
    build.build()
    binding.lib()
    return binding
