import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (a GB300, sm_103a)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built for sm_103a, loaded through the Python binding."""
    from deepseek_moe_layer_gb300 import binding
    return binding.lib()
