"""sbgemm_noalloc, the entry point for callers that cannot allocate device
memory: code running under CUDA graph capture (where cudaMalloc is not
allowed), plugins that are handed only their input and output buffers, loops
that must not pay cudaMalloc's synchronisation, and runtimes whose allocator
owns the whole device.  It runs the split schedules on the library's own
static scratch array instead of a caller workspace.

Each case is checked on two calls in a row (the array keeps the previous
call's contents, so flags and counters must be cleared before every launch):
against the oracle within the fp32 bound (exactly on integer inputs), and bit
for bit against sbgemm_ex given the same options and a caller workspace of the
same size.  The cases cover both uses of the scratch on the TMA path (chained
stream-K over the last waves, independent K pieces of few-tile long-K
products) and the gather path's K pieces of a small product.  Between the two
calls neither torch's allocator nor the device's free memory may change.

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
    # (M, N, K, batch, a_layout, b_layout, accumulate, values, schedule)
    (2048, 2560, 1024, 1, "row16", "col16", 0, "real", sg.STREAM_K_CHAINED),
    (1024, 1024, 768, 5, "col16", "row16", 1, "real", sg.STREAM_K_CHAINED),
    (2048, 2600, 1000, 1, "row16", "row16", 1, "int", sg.STREAM_K_CHAINED),
    (1280, 1024, 4096, 1, "row16", "col16", 1, "real", sg.STREAM_K_PIECES),
    (2048, 640, 5000, 1, "col16", "row16", 0, "int", sg.STREAM_K_PIECES),
]


def _args(case, dA, dB, dC, torch):
    return (dA.data_ptr() + 4 * case.A.offset, case.A.rs, case.A.cs, case.A.bs,
            dB.data_ptr() + 4 * case.B.offset, case.B.rs, case.B.cs, case.B.bs,
            dC.data_ptr() + 4 * case.C.offset, case.C.rs, case.C.cs, case.C.bs,
            case.M, case.N, case.K, case.batch, case.alpha, case.accumulate,
            torch.cuda.current_stream().cuda_stream)


def _check_twice(torch, case, want_schedule, want_path=None):
    dA, dB = gu.to_device(case.A, torch), gu.to_device(case.B, torch)
    # The regular entry point, same options, a caller workspace of the same size.
    ws = torch.empty(sg.NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
    dC = torch.from_numpy(case.C.storage.copy()).to("cuda")
    args = _args(case, dA, dB, dC, torch)
    plan = sg.sbgemm_plan(*args[:16], case.accumulate, workspace=ws.data_ptr(),
                          workspace_bytes=ws.numel(), k_split=sg.KSPLIT_ANY)
    assert plan["stream_k"] == want_schedule, plan
    if want_path is not None:
        assert plan["path_name"] == want_path, plan
    sg.sbgemm_ex(*args, workspace=ws.data_ptr(), workspace_bytes=ws.numel(),
                 k_split=sg.KSPLIT_ANY)
    torch.cuda.synchronize()
    want = gu.logical_c(case, dC.cpu().numpy())

    ref, bound = oracle.case_product(case)
    exact = case.values == "int"
    for call in range(2):
        dC2 = torch.from_numpy(case.C.storage.copy()).to("cuda")
        torch.cuda.synchronize()
        alloc0 = torch.cuda.memory_allocated()
        free0 = torch.cuda.mem_get_info()[0]
        sg.sbgemm_noalloc(*_args(case, dA, dB, dC2, torch))
        torch.cuda.synchronize()
        if call == 1:
            # The first call on a device may look up the scratch's address;
            # the second allocates nothing anywhere.
            assert torch.cuda.memory_allocated() == alloc0
            assert torch.cuda.mem_get_info()[0] == free0
        got = gu.logical_c(case, dC2.cpu().numpy())
        diff = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
        assert diff.size == 0, (f"call {call}: {len(diff)} elements differ from sbgemm_ex, "
                                f"first {tuple(diff[0])}")
        g64 = got.astype(np.float64)
        if exact:
            bad = np.argwhere(g64 != ref.astype(np.float32).astype(np.float64))
        else:
            bad = np.argwhere(~(np.abs(g64 - ref) <= gu.TOL_FFMA * bound))
        assert bad.size == 0, f"call {call}: {len(bad)} elements off the oracle, first {tuple(bad[0])}"
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where


@pytest.mark.parametrize("shape", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}b{c[3]}" for c in CASES])
def test_no_alloc_matches_regular_entry_point_twice(torch, shape):
    M, N, K, batch, la, lb, acc, values, schedule = shape
    rng = np.random.default_rng(M + 7 * N + K)
    case = wl.random_strided(rng, M, N, K, batch, la, lb, values=values, accumulate=acc,
                             alpha=0.5)
    _check_twice(torch, case, schedule, want_path="tma_ffma")


@pytest.mark.parametrize("values", ["real", "int"])
def test_no_alloc_gather_k_pieces_twice(torch, values):
    # The MLP layer 256 x 784 -> 512: 32 tiles of 64 x 64 on the gather path,
    # each cut into K pieces that the scratch holds.
    case = wl.make("c2a", values)
    _check_twice(torch, case, sg.STREAM_K_PIECES, want_path="gather_ffma")
