import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # A gpu-marked test on a machine without a GPU fails loudly instead of
    # skipping: a skipped device test must not read as a pass.
    pass


@pytest.fixture(autouse=True)
def _device_status_after_each_gpu_test(request):
    """With SBGEMM_CHECK_STATUS=1 (the debug-build run), every GPU test must
    leave the device status words clean: no bounded wait ran out and no
    bounds check of the debug build fired."""
    yield
    if os.environ.get("SBGEMM_CHECK_STATUS") == "1" and request.node.get_closest_marker("gpu"):
        import strided_gemm_gb300 as sg
        st, where = sg.sbgemm_device_status()
        assert st == sg.SBGEMM_OK, f"device status {st} (code {where}) after {request.node.nodeid}"


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()
