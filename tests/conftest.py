import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle
    _oracle.build()
    return _oracle


@pytest.fixture(autouse=True)
def _bounds_checked_error_word(request):
    """Under EXL3_BOUNDS_CHECKED=1 (the bounds-checked library), every GPU test
    must leave the device error word free of bounds and timeout errors."""
    yield
    if os.environ.get("EXL3_BOUNDS_CHECKED") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import trellis_quantized_linear_gb300 as tql
    if tql._lib is None:
        return
    status = tql.exl3_get_device_status()
    assert status not in (7, 9), f"device error word after {request.node.nodeid}: {tql.STATUS_NAMES.get(status)}"
