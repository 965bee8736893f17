"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies gives up after a short limit, records where, and the kernel returns.
The host reads SBGEMM_ERR_DEVICE_TIMEOUT and the context stays usable."""

import numpy as np
import pytest

import strided_gemm_gb300 as sg
import workloads as wl
from strided_gemm_gb300 import build as sgbuild
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    sgbuild.build()
    sg.load()
    return t


@pytest.mark.parametrize("what,code", [(sg.SELFTEST_MBARRIER, 7), (sg.SELFTEST_FLAG, 8)],
                         ids=["mbarrier", "flag"])
def test_bounded_wait_runs_out_and_context_survives(torch, what, code):
    assert sg.sbgemm_device_status() == (sg.SBGEMM_OK, 0)
    sg.sbgemm_selftest(what, 20000)          # 20 ms
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_ERR_DEVICE_TIMEOUT and where == code
    # Read once, cleared.
    assert sg.sbgemm_device_status() == (sg.SBGEMM_OK, 0)
    # The context is still usable: a normal product is exact.
    case = wl.make("c1", "int")
    got = gu.run_case(case, torch)
    gu.check_full(case, got, exact=True)
    assert sg.sbgemm_device_status() == (sg.SBGEMM_OK, 0)


def test_selftest_rejects_bad_arguments(torch):
    for what, limit in ((0, 10), (3, 10), (1, 0), (1, 3_000_000)):
        with pytest.raises(sg.SbgemmError) as e:
            sg.sbgemm_selftest(what, limit)
        assert e.value.status == sg.SBGEMM_ERR_INVALID_VALUE
