import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """Around every GPU test: the device status word starts clear and, after the
    test, holds no record of an access outside a buffer.  (Only the library
    built with MX_BOUNDS_CHECK=1 records those; there, this turns every GPU test
    into a bounds check of the kernels it ran.)"""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import block_scaled_fp4_bf16_gb300 as mx
    mx.mx_device_status()
    yield
    rc = mx.mx_device_status()
    assert rc != mx.MX_ERR_DEVICE_BOUNDS, (
        f"{request.node.nodeid}: a kernel accessed memory outside a buffer "
        f"({mx.mx_last_error_string()})")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle
    _oracle.build()
    return _oracle
