"""Full-size products compared with the oracle at every element (the StaleyNET
"GPU Implementation" page, section "Testing the kernels": each output against
a plain CPU implementation of the same formula).  One case per kernel and
schedule, through the call a caller with a workspace makes:

- TMA-fed FFMA, chained stream-K over the last waves (c5a, real and integer;
  c5b, whose half-full last tile column is split by weighted cost);
- TMA-fed FFMA, independent K pieces of a few-tile long-K product (f1dwa);
- TMA-fed FFMA, data-parallel over a batch of 128 (c3) and the 512 x 64
  tiles of a narrow accumulating product (c4);
- strided gather, K pieces of a small product (c2a), and the 128 x 64 tiles
  of the spectrogram's overlapping frames (f4spec);
- TF32 tensor cores, the transposed plan with split K (c5c, real and
  integer) and both operands MN-major with split K (f1dwb).

Real values must lie within the problem's bound (1e-5, or 2e-3 on TF32, times
|alpha| sum_k |a||b| + |C0|); integer values must match bit for bit."""

import numpy as np
import pytest

import oracle
import strided_gemm_gb300 as sg
import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need a CUDA device"
    sg.load()
    return t


@pytest.fixture(scope="module")
def workspace(torch):
    return torch.empty(sg.sbgemm_workspace_bytes(torch.cuda.current_device()), dtype=torch.uint8,
                       device="cuda")


CASES = [
    # (workload, values, math, path, stream_k schedule)
    ("c5a", "real", sg.MATH_FP32, "tma_ffma", sg.STREAM_K_CHAINED),
    ("c5a", "int", sg.MATH_FP32, "tma_ffma", sg.STREAM_K_CHAINED),
    ("c5b", "real", sg.MATH_FP32, "tma_ffma", sg.STREAM_K_CHAINED),
    ("f1dwa", "real", sg.MATH_FP32, "tma_ffma", sg.STREAM_K_PIECES),
    ("c3", "real", sg.MATH_FP32, "tma_ffma", sg.STREAM_K_NONE),
    ("c4", "real", sg.MATH_FP32, "tma_ffma", sg.STREAM_K_NONE),
    ("c2a", "real", sg.MATH_FP32, "gather_ffma", sg.STREAM_K_PIECES),
    ("f4spec", "real", sg.MATH_FP32, "gather_ffma", sg.STREAM_K_NONE),
    ("c5c", "real", sg.MATH_TF32, "tma_tf32", sg.STREAM_K_PIECES),
    ("c5c", "int", sg.MATH_TF32, "tma_tf32", sg.STREAM_K_PIECES),
    ("f1dwb", "real", sg.MATH_TF32, "tma_tf32", sg.STREAM_K_PIECES),
]


@pytest.mark.parametrize("name,values,math,path,schedule", CASES,
                         ids=[f"{c[0]}-{c[1]}-{'tf32' if c[2] else 'fp32'}" for c in CASES])
def test_full_size_every_element(torch, workspace, name, values, math, path, schedule):
    case = wl.make(name, values)
    dA, dB = gu.to_device(case.A, torch), gu.to_device(case.B, torch)
    dC = torch.from_numpy(case.C.storage.copy()).to("cuda")
    args = (dA.data_ptr() + 4 * case.A.offset, case.A.rs, case.A.cs, case.A.bs,
            dB.data_ptr() + 4 * case.B.offset, case.B.rs, case.B.cs, case.B.bs,
            dC.data_ptr() + 4 * case.C.offset, case.C.rs, case.C.cs, case.C.bs,
            case.M, case.N, case.K, case.batch, case.alpha, case.accumulate,
            torch.cuda.current_stream().cuda_stream)
    kw = dict(math=math, workspace=workspace.data_ptr(), workspace_bytes=workspace.numel())
    plan = sg.sbgemm_plan(*args[:16], case.accumulate, **kw)
    assert plan["path_name"] == path and plan["stream_k"] == schedule, plan
    if name == "f4spec":
        assert (plan["tile_m"], plan["tile_n"]) == (128, 64), plan
    sg.sbgemm_ex(*args, **kw)
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    st, where = sg.sbgemm_device_status()
    assert st == sg.SBGEMM_OK, where
    tol = gu.TOL_TF32 if math == sg.MATH_TF32 else gu.TOL_FFMA
    gu.check_full(case, got, tol=tol, exact=(values == "int"))
