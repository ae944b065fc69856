import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


@pytest.fixture(scope="session", autouse=True)
def _built_library(request):
    """Build libmoeq.so once per session when any GPU test is collected."""
    if any(item.get_closest_marker("gpu") for item in request.session.items):
        from weight_quantized_moe_gb300 import build
        build.build()
    yield
