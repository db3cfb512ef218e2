import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


import pytest


@pytest.fixture
def opt():
    """Sets library options (nvfp4_set_option) for one test and puts back the
    previous values afterwards."""
    from nvfp4_quantized_matmul_gb300 import binding

    saved = {}

    def set_(name, value):
        if name not in saved:
            saved[name] = binding.get_option(name)
        binding.set_option(name, value)

    yield set_
    for name, value in saved.items():
        binding.set_option(name, value)
