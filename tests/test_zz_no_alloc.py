"""sbgemm_noalloc, the entry point for callers that cannot allocate device
memory (graph-capture regions, plugins given only their input and output
buffers, loops that must not synchronise on cudaMalloc).  It runs the stream-K
schedule on the library's own static scratch; its results must match the
regular entry point fed a caller-owned workspace, on two calls in a row (the
scratch keeps the previous call's contents, and its flags must be cleared
before each launch).

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import numpy as np
import pytest

import oracle
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


CASES = [
    # (M, N, K, batch, a_layout, b_layout, accumulate, values): each plans stream-K
    (2048, 2560, 1024, 1, "row16", "col16", 0, "real"),
    (1024, 1024, 768, 5, "col16", "row16", 1, "real"),
    (2048, 2600, 1000, 1, "row16", "row16", 1, "int"),
]


def _args(case, dA, dB, dC, torch):
    return (dA.data_ptr() + 4 * case.A.offset, case.A.rs, case.A.cs, case.A.bs,
            dB.data_ptr() + 4 * case.B.offset, case.B.rs, case.B.cs, case.B.bs,
            dC.data_ptr() + 4 * case.C.offset, case.C.rs, case.C.cs, case.C.bs,
            case.M, case.N, case.K, case.batch, case.alpha, case.accumulate,
            torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}b{c[3]}" for c in CASES])
def test_no_alloc_matches_regular_entry_point_twice(torch, shape):
    M, N, K, batch, la, lb, acc, values = shape
    rng = np.random.default_rng(M + 7 * N + K)
    case = wl.random_strided(rng, M, N, K, batch, la, lb, values=values, accumulate=acc,
                             alpha=0.5)
    dA, dB = gu.to_device(case.A, torch), gu.to_device(case.B, torch)

    # The regular entry point with a caller-owned workspace.
    ws = torch.empty(sg.sbgemm_workspace_bytes(torch.cuda.current_device()),
                     dtype=torch.uint8, device="cuda")
    dC = torch.from_numpy(case.C.storage.copy()).to("cuda")
    args = _args(case, dA, dB, dC, torch)
    plan = sg.sbgemm_plan(*args[:16], case.accumulate, workspace=ws.data_ptr(),
                          workspace_bytes=ws.numel())
    assert plan["stream_k"], "the case must exercise the scratch"
    sg.sbgemm_ex(*args, workspace=ws.data_ptr(), workspace_bytes=ws.numel())
    torch.cuda.synchronize()
    want = gu.logical_c(case, dC.cpu().numpy()).astype(np.float64)

    _, bound = oracle.case_product(case)
    for call in range(2):
        dC2 = torch.from_numpy(case.C.storage.copy()).to("cuda")
        sg.sbgemm_noalloc(*_args(case, dA, dB, dC2, torch))
        torch.cuda.synchronize()
        got = gu.logical_c(case, dC2.cpu().numpy()).astype(np.float64)
        bad = np.argwhere(~(np.abs(got - want) <= gu.TOL_FFMA * bound))
        assert bad.size == 0, f"call {call}: {len(bad)} elements differ, first {tuple(bad[0])}"
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where
